// paged_attention_forward_static_ws: the forward call for callers that cannot
// allocate device memory.
//
// Some callers have no way to hand this library a workspace: code running
// under a custom or fixed-budget allocator that forbids new device
// allocations after start-up, runtimes that only pass through
// already-registered buffers, or plugin hosts whose memory is owned
// elsewhere.  For them this entry point uses a scratch area that lives in
// the library itself: a file-scope __device__ array of
// kStaticWorkspaceBytes, which every GPU that loads the library holds until
// the process exits.  Nothing is allocated per call; the caller still passes
// its inputs and output.
//
// The scratch holds the planner's work lists and the split-KV partial rows.
// The planner rewrites everything a call reads (counters included) before the
// attention kernels run, so stale contents from an earlier call are harmless.
// All calls on a device share the one array: calls whose GPU work overlaps
// (different streams, or different host threads without ordering) race on it.
#include <cuda_runtime.h>

#include <stdio.h>

#include "paged_kv.h"
#include "pkv_internal.h"

namespace {

constexpr size_t kStaticWorkspaceBytes = size_t(8) << 20;  // 8 MiB per device

static __device__ __align__(256) unsigned char g_static_workspace[kStaticWorkspaceBytes];

// Device address of the scratch on the current device.  In host code
// g_static_workspace names a host-side stand-in, not device memory, so the
// address is looked up with that device current: on every call, which costs
// a runtime query and allocates nothing, so that an address never outlives
// the module it came from (after cudaDeviceReset the library's device module
// is loaded again, at another address).
pkv_status static_scratch(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    pkv::set_last_error("static scratch: no usable current device");
    return PKV_ERR_CUDA;
  }
  void* p = nullptr;
  e = cudaGetSymbolAddress(&p, g_static_workspace);
  if (e != cudaSuccess || !p) {
    pkv::set_last_error("static scratch: cudaGetSymbolAddress failed");
    return PKV_ERR_CUDA;
  }
  *out = p;
  return PKV_OK;
}

}  // namespace

extern "C" {

size_t paged_attention_static_workspace_bytes(void) { return kStaticWorkspaceBytes; }

pkv_status paged_attention_forward_static_ws(const void* q, const void* k_cache, const void* v_cache,
                                             const int32_t* block_tables, const int32_t* context_lens,
                                             const int32_t* query_start_loc, void* out, int32_t num_seqs,
                                             int64_t num_tokens, int32_t num_q_heads, int32_t num_kv_heads,
                                             int32_t head_dim, int64_t num_blocks, int32_t block_size,
                                             int32_t max_blocks_per_seq, int32_t max_query_len, float scale,
                                             int32_t causal, int32_t hints, pkv_dtype dtype, void* stream) {
  const size_t need = paged_attention_workspace_min(num_seqs, num_tokens, num_q_heads, num_kv_heads, head_dim);
  if (need > kStaticWorkspaceBytes) {
    char msg[200];
    snprintf(msg, sizeof(msg), "batch needs %zu bytes of scratch; the built-in static scratch holds %zu", need,
             kStaticWorkspaceBytes);
    pkv::set_last_error(msg);
    return PKV_ERR_WORKSPACE;
  }
  void* ws = nullptr;
  const pkv_status st = static_scratch(&ws);
  if (st != PKV_OK) return st;
  return paged_attention_forward(q, k_cache, v_cache, block_tables, context_lens, query_start_loc, out, num_seqs,
                                 num_tokens, num_q_heads, num_kv_heads, head_dim, num_blocks, block_size,
                                 max_blocks_per_seq, max_query_len, scale, causal, hints, ws, kStaticWorkspaceBytes,
                                 dtype, stream);
}

}  // extern "C"
