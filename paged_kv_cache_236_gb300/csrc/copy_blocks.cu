// Copy-on-write of whole blocks of the device pool (paged_kv_copy_blocks,
// declared in paged_kv_blocks.h).
//
// Dao-AILab/flash-attention issue #660: the cache manager copies and updates
// the pages.  When a sequence appends to a partly filled block that another
// block table also names, the host block manager gives it a fresh block and a
// (src, dst) pair; this copies block src onto block dst in every layer's K
// and V pool before the step's new rows are written.
//
// The pairs come from host memory and travel in the launch parameters
// (kPairsPerLaunch per launch, so no host-to-device copy and no device-side
// id check: ids are checked on the host before any launch).  HBM-bound:
// a work unit (pair, layer, K or V) copies one block, 16-byte chunks, four
// per thread in flight; sources are never destinations in one call, so the
// loads take the read-only path.
#include <cuda_runtime.h>

#include <stdint.h>
#include <stdio.h>

#include <unordered_set>

#include "paged_kv_blocks.h"
#include "pkv_internal.h"

namespace {

constexpr int kPairsPerLaunch = 4000;  // 32 000 bytes: parameters stay under the 32 764-byte limit
constexpr int kMaxGrid = 1024;

struct CopyList {
  int n;
  int32_t pair[2 * kPairsPerLaunch];
};

__device__ __forceinline__ int4 ld_stream(const int4* p) {
  int4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.s32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

__global__ void __launch_bounds__(256) copy_blocks_kernel(uint8_t* kc, uint8_t* vc, const __grid_constant__ CopyList list,
                                                          int layers, int64_t layer_stride_b, int block_chunks) {
  const int n_units = list.n * layers * 2;
  for (int w = blockIdx.x; w < n_units; w += gridDim.x) {
    const int pair = w / (2 * layers), r = w - pair * 2 * layers;
    const int layer = r >> 1, kv = r & 1;
    const int64_t src = list.pair[2 * pair], dst = list.pair[2 * pair + 1];
    uint8_t* base = (kv ? vc : kc) + layer * layer_stride_b;
    const int4* s = reinterpret_cast<const int4*>(base + src * block_chunks * 16);
    int4* d = reinterpret_cast<int4*>(base + dst * block_chunks * 16);
    for (int c0 = threadIdx.x; c0 < block_chunks; c0 += 4 * blockDim.x) {
      int4 v[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int c = c0 + i * blockDim.x;
        if (c < block_chunks) v[i] = ld_stream(s + c);
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int c = c0 + i * blockDim.x;
        if (c < block_chunks) d[c] = v[i];
      }
    }
  }
}

pkv_status fail(pkv_status st, const char* msg, long long a = 0) {
  char buf[256];
  snprintf(buf, sizeof(buf), msg, a);
  pkv::set_last_error(buf);
  return st;
}

}  // namespace

extern "C" pkv_status paged_kv_copy_blocks(void* k_cache, void* v_cache, const int32_t* copies, int32_t num_copies,
                                           int32_t num_layers, int64_t layer_stride, int64_t num_blocks,
                                           int32_t block_size, int32_t num_kv_heads, int32_t head_dim,
                                           pkv_dtype dtype, void* stream) {
  pkv::set_last_error("");
  if (dtype != PKV_DTYPE_BF16 && dtype != PKV_DTYPE_F32) return fail(PKV_ERR_UNSUPPORTED, "dtype %lld", (int)dtype);
  if (num_copies < 0 || num_layers <= 0 || num_blocks <= 0 || block_size <= 0 || num_kv_heads <= 0 || head_dim <= 0)
    return fail(PKV_ERR_INVALID_ARG, "sizes must be positive (num_copies >= 0)");
  const int64_t eb = dtype == PKV_DTYPE_BF16 ? 2 : 4;
  const int64_t block_elems = (int64_t)block_size * num_kv_heads * head_dim;
  if (block_elems * eb % 16 != 0) return fail(PKV_ERR_UNSUPPORTED, "block bytes not a multiple of 16");
  if (block_elems * eb / 16 > ((int64_t)1 << 30)) return fail(PKV_ERR_UNSUPPORTED, "blocks too large");
  if (num_blocks > ((int64_t)1 << 31) - 1) return fail(PKV_ERR_UNSUPPORTED, "num_blocks exceeds int32");
  if (layer_stride == 0) layer_stride = num_blocks * block_elems;
  if (layer_stride < num_blocks * block_elems) return fail(PKV_ERR_INVALID_ARG, "layer_stride smaller than one pool");
  if (layer_stride * eb % 16 != 0) return fail(PKV_ERR_INVALID_ARG, "layer stride bytes not a multiple of 16");
  if ((int64_t)num_layers * 2 * kPairsPerLaunch > ((int64_t)1 << 31) - 1)
    return fail(PKV_ERR_UNSUPPORTED, "num_layers too large");
  if (num_copies == 0) return PKV_OK;
  if (!k_cache || !v_cache || !copies) return fail(PKV_ERR_INVALID_ARG, "null pointer");
  if ((reinterpret_cast<uintptr_t>(k_cache) | reinterpret_cast<uintptr_t>(v_cache)) & 15u)
    return fail(PKV_ERR_INVALID_ARG, "caches must be 16-byte aligned");
  // ids in range; no destination is a source or repeats
  std::unordered_set<int32_t> dsts;
  for (int32_t i = 0; i < num_copies; ++i) {
    const int32_t s = copies[2 * i], d = copies[2 * i + 1];
    if (s < 0 || s >= num_blocks || d < 0 || d >= num_blocks)
      return fail(PKV_ERR_INVALID_ARG, "copy pair %lld names a block outside the pool", i);
    if (!dsts.insert(d).second) return fail(PKV_ERR_INVALID_ARG, "block %lld is a destination twice", d);
  }
  for (int32_t i = 0; i < num_copies; ++i)
    if (dsts.count(copies[2 * i])) return fail(PKV_ERR_INVALID_ARG, "block %lld is a source and a destination",
                                               copies[2 * i]);
  const int block_chunks = (int)(block_elems * eb / 16);
  static thread_local CopyList list;  // 32 KB: off the stack
  for (int32_t first = 0; first < num_copies; first += kPairsPerLaunch) {
    const int n = num_copies - first < kPairsPerLaunch ? num_copies - first : kPairsPerLaunch;
    list.n = n;
    for (int i = 0; i < 2 * n; ++i) list.pair[i] = copies[2 * first + i];
    const int units = n * num_layers * 2;
    const int grid = units < kMaxGrid ? units : kMaxGrid;
    copy_blocks_kernel<<<grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<uint8_t*>(k_cache), static_cast<uint8_t*>(v_cache), list, num_layers, layer_stride * eb,
        block_chunks);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
      char buf[256];
      snprintf(buf, sizeof(buf), "paged_kv_copy_blocks launch: %s", cudaGetErrorString(e));
      pkv::set_last_error(buf);
      return PKV_ERR_CUDA;
    }
  }
  return PKV_OK;
}
