// Host side of the C ABI declared in include/paged_kv.h: argument checks,
// tensor-map encoding, workspace layout and the launch sequence
//   planner -> tensor-core kernel (multi-token rows) -> CUDA-core kernel
//   (decode-shaped rows)
// all on the caller's stream, with no host synchronisation (split-KV partial
// rows are merged inside the attention kernels by the last split to finish).
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <math.h>
#include <algorithm>
#include <mutex>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include "paged_kv.h"
#include "pkv_internal.h"

namespace {

thread_local char g_msg[512] = "";
thread_local cudaEvent_t g_prof_start = nullptr, g_prof_stop = nullptr, g_prof_mid = nullptr;
// pkv_debug_fault: armed for the next forward call of this thread only
thread_local int g_fault_tile = 0;
thread_local uint64_t g_fault_wait_ns = 0;

pkv_status fail(pkv_status st, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
  va_end(ap);
  return st;
}

pkv_status cuda_fail(cudaError_t e, const char* what) {
  return fail(PKV_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

// Sticky device error word: one per device (a __device__ variable exists on
// every device that loads this library).
__device__ int g_device_error;

struct DeviceInfo {
  bool ready = false;
  int sms = 0;
  int major = 0, minor = 0;
  int* err = nullptr;  // device address of g_device_error
};

std::mutex g_mu;
DeviceInfo g_dev[64];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

pkv_status device_info(DeviceInfo** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= 64) return fail(PKV_ERR_UNSUPPORTED, "device ordinal %d out of range", dev);
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceInfo& d = g_dev[dev];
  if (!d.ready) {
    if ((e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
      return cuda_fail(e, "cudaDeviceGetAttribute");
    cudaDeviceGetAttribute(&d.major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&d.minor, cudaDevAttrComputeCapabilityMinor, dev);
    if (!(d.major == 10 && d.minor == 3))
      return fail(PKV_ERR_UNSUPPORTED, "this library is built for sm_103a; device %d is sm_%d%d", dev, d.major,
                  d.minor);
    void* p = nullptr;
    if ((e = cudaGetSymbolAddress(&p, g_device_error)) != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress");
    d.err = static_cast<int*>(p);
    if (!g_encode) {
      void* fn = nullptr;
      cudaDriverEntryPointQueryResult q;
      e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
      if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn)
        return fail(PKV_ERR_CUDA, "cuTensorMapEncodeTiled entry point unavailable");
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    d.ready = true;
  }
  *out = &d;
  return PKV_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int elem_bytes(pkv_dtype dt) { return dt == PKV_DTYPE_BF16 ? 2 : dt == PKV_DTYPE_FP8_E4M3 ? 1 : 4; }

// 4-D map of a block pool [NB, bs, Hkv, D] with a box of one block of one kv head.
pkv_status encode_pool_map(CUtensorMap* map, const void* base, pkv_dtype dt, int64_t NB, int bs, int Hkv, int D,
                           int box_d, CUtensorMapSwizzle swz) {
  const int es = elem_bytes(dt);
  cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)Hkv, (cuuint64_t)bs, (cuuint64_t)NB};
  cuuint64_t strides[3] = {(cuuint64_t)D * es, (cuuint64_t)Hkv * D * es, (cuuint64_t)bs * Hkv * D * es};
  cuuint32_t box[4] = {(cuuint32_t)box_d, 1, (cuuint32_t)bs, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUtensorMapDataType ty = dt == PKV_DTYPE_BF16        ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                 : dt == PKV_DTYPE_FP8_E4M3 ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                                            : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
  CUresult r = g_encode(map, ty,
                        4, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(PKV_ERR_CUDA, "cuTensorMapEncodeTiled (pool) failed: %d", (int)r);
  return PKV_OK;
}

// 3-D map of q [T, Hq, D] with a box of {box_d, G heads, tokens}.
pkv_status encode_q_map(CUtensorMap* map, const void* base, int64_t T, int Hq, int D, int box_d, int G, int tokens) {
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)Hq, (cuuint64_t)(T > 0 ? T : 1)};
  cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)Hq * D * 2};
  cuuint32_t box[3] = {(cuuint32_t)box_d, (cuuint32_t)G, (cuuint32_t)tokens};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(PKV_ERR_CUDA, "cuTensorMapEncodeTiled (q) failed: %d", (int)r);
  return PKV_OK;
}

constexpr size_t kAlign = 256;
size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

// Item-count targets used for capacity sizing (device-independent upper
// bounds of the per-device targets below).
constexpr int kCapTargetDec = 4096;
constexpr int kCapTargetMma = 2048;
constexpr int kDefaultPartRows = 32768;

}  // namespace

namespace pkv {

void set_last_error(const char* msg) { snprintf(g_msg, sizeof(g_msg), "%s", msg); }

WorkspaceLayout workspace_layout(int B, int64_t T, int Hq, int Hkv, int D, size_t bytes_available, int /*num_sms*/,
                                 bool want_default_parts) {
  WorkspaceLayout L{};
  const int G = Hq / Hkv;
  const int64_t rows = T * (int64_t)G;
  const int64_t dec_units = (int64_t)Hkv * ((rows + kDecRows - 1) / kDecRows + B);
  // tensor-core items hold whole tokens: floor(kMmaRows / G) of them
  const int64_t mma_tok = G <= kMmaRows ? kMmaRows / G : 1;
  const int64_t mma_units = (int64_t)Hkv * ((T + mma_tok - 1) / mma_tok + B);
  const int64_t dec_cap = kCapTargetDec + dec_units;
  const int64_t mma_cap = kCapTargetMma + mma_units;
  const int64_t merge_cap = dec_cap + mma_cap;
  size_t off = 0;
  L.header_off = off;
  off = align_up(off + sizeof(PlanHeader));
  L.dec_off = off;
  off = align_up(off + (size_t)dec_cap * sizeof(WorkItem));
  L.mma_off = off;
  off = align_up(off + (size_t)mma_cap * sizeof(WorkItem));
  L.merge_off = off;
  off = align_up(off + (size_t)merge_cap * sizeof(MergeGroup));
  L.ticket_off = off;
  off = align_up(off + (size_t)merge_cap * sizeof(int));
  L.seq_off = off;  // per-sequence planner scratch: prefix keys, group, tile-match mask
  off = align_up(off + (size_t)B * 4 * sizeof(int));
  L.pre_off = off;  // prefix groups (at most one per sequence)
  off = align_up(off + (size_t)B * sizeof(PreGroup));
  const size_t fixed = off;
  const size_t per_row = sizeof(float2) + (size_t)D * sizeof(float);
  int64_t part_cap = 0;
  if (want_default_parts) {
    part_cap = kDefaultPartRows;
  } else if (bytes_available > fixed + 2 * kAlign) {
    part_cap = (int64_t)((bytes_available - fixed - 2 * kAlign) / per_row);
    if (part_cap > (int64_t)1 << 30) part_cap = (int64_t)1 << 30;
  }
  L.ml_off = off;
  off = align_up(off + (size_t)part_cap * sizeof(float2));
  L.acc_off = off;
  off = align_up(off + (size_t)part_cap * D * sizeof(float));
  L.total = part_cap > 0 ? off : fixed;
  L.dec_cap = (int)dec_cap;
  L.mma_cap = (int)mma_cap;
  L.merge_cap = (int)merge_cap;
  L.part_cap = (int)part_cap;
  return L;
}

}  // namespace pkv

using namespace pkv;

extern "C" {

const char* pkv_last_error(void) { return g_msg; }

const char* pkv_version(void) { return "paged_kv 0.1.0 sm_103a"; }

void pkv_set_profile_events(void* start, void* stop) {
  g_prof_start = static_cast<cudaEvent_t>(start);
  g_prof_stop = static_cast<cudaEvent_t>(stop);
  if (!g_prof_start || !g_prof_stop) g_prof_start = g_prof_stop = nullptr;
}

void pkv_set_profile_mid_event(void* mid) { g_prof_mid = static_cast<cudaEvent_t>(mid); }

pkv_status pkv_event_elapsed_ms(void* start, void* stop, float* ms) {
  if (!start || !stop || !ms) return fail(PKV_ERR_INVALID_ARG, "null argument");
  cudaError_t e = cudaEventElapsedTime(ms, static_cast<cudaEvent_t>(start), static_cast<cudaEvent_t>(stop));
  if (e != cudaSuccess) return cuda_fail(e, "cudaEventElapsedTime");
  return PKV_OK;
}

pkv_status pkv_debug_fault(int32_t fault_tile, int64_t wait_ns) {
  if (fault_tile < 0 || wait_ns < 0) return fail(PKV_ERR_INVALID_ARG, "fault_tile and wait_ns must be >= 0");
  g_fault_tile = fault_tile;
  g_fault_wait_ns = (uint64_t)wait_ns;
  return PKV_OK;
}

pkv_status pkv_device_errors(int32_t* flags, int32_t clear) {
  if (!flags) return fail(PKV_ERR_INVALID_ARG, "flags is NULL");
  DeviceInfo* d = nullptr;
  pkv_status st = device_info(&d);
  if (st != PKV_OK) return st;
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
  int v = 0;
  if ((e = cudaMemcpy(&v, d->err, sizeof(int), cudaMemcpyDeviceToHost)) != cudaSuccess)
    return cuda_fail(e, "read device error word");
  if (clear) {
    const int z = 0;
    if ((e = cudaMemcpy(d->err, &z, sizeof(int), cudaMemcpyHostToDevice)) != cudaSuccess)
      return cuda_fail(e, "clear device error word");
  }
  *flags = v;
  return PKV_OK;
}

pkv_status paged_kv_write(const void* k, const void* v, const int64_t* slot_mapping, void* k_cache, void* v_cache,
                          int64_t num_tokens, int64_t num_blocks, int32_t block_size, int32_t num_kv_heads,
                          int32_t head_dim, int64_t k_token_stride, int64_t v_token_stride, pkv_dtype dtype,
                          void* stream) {
  g_msg[0] = 0;
  if (dtype != PKV_DTYPE_BF16 && dtype != PKV_DTYPE_F32) return fail(PKV_ERR_UNSUPPORTED, "dtype %d", (int)dtype);
  if (num_tokens < 0 || num_blocks <= 0 || block_size <= 0 || num_kv_heads <= 0 || head_dim <= 0)
    return fail(PKV_ERR_INVALID_ARG, "sizes must be positive (num_tokens >= 0)");
  const int64_t row = (int64_t)num_kv_heads * head_dim;
  if (row > (1 << 24)) return fail(PKV_ERR_UNSUPPORTED, "num_kv_heads * head_dim too large");
  if (k_token_stride == 0) k_token_stride = row;
  if (v_token_stride == 0) v_token_stride = row;
  if (k_token_stride < row || v_token_stride < row)
    return fail(PKV_ERR_INVALID_ARG, "token stride smaller than num_kv_heads * head_dim");
  if (num_tokens == 0) return PKV_OK;
  if (!k || !v || !slot_mapping || !k_cache || !v_cache) return fail(PKV_ERR_INVALID_ARG, "null pointer");
  if (!aligned16(k_cache) || !aligned16(v_cache)) return fail(PKV_ERR_INVALID_ARG, "caches must be 16-byte aligned");
  DeviceInfo* d = nullptr;
  pkv_status st = device_info(&d);
  if (st != PKV_OK) return st;
  cudaError_t e = launch_kv_write(k, v, slot_mapping, k_cache, v_cache, num_tokens, num_blocks * block_size,
                                  (int)row, elem_bytes(dtype), k_token_stride, v_token_stride, d->err,
                                  static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "paged_kv_write launch");
  return PKV_OK;
}

pkv_status paged_kv_write_fp8(const void* k, const void* v, const int64_t* slot_mapping, void* k_cache,
                              void* v_cache, int64_t num_tokens, int64_t num_blocks, int32_t block_size,
                              int32_t num_kv_heads, int32_t head_dim, int64_t k_token_stride, int64_t v_token_stride,
                              pkv_dtype dtype, float k_scale, float v_scale, void* stream) {
  g_msg[0] = 0;
  if (dtype != PKV_DTYPE_BF16 && dtype != PKV_DTYPE_F32) return fail(PKV_ERR_UNSUPPORTED, "dtype %d", (int)dtype);
  if (num_tokens < 0 || num_blocks <= 0 || block_size <= 0 || num_kv_heads <= 0 || head_dim <= 0)
    return fail(PKV_ERR_INVALID_ARG, "sizes must be positive (num_tokens >= 0)");
  if (!(k_scale > 0.f) || !isfinite(k_scale) || !(v_scale > 0.f) || !isfinite(v_scale))
    return fail(PKV_ERR_INVALID_ARG, "k_scale and v_scale must be positive and finite");
  const int64_t row = (int64_t)num_kv_heads * head_dim;
  if (row > (1 << 24)) return fail(PKV_ERR_UNSUPPORTED, "num_kv_heads * head_dim too large");
  if (row % 16 != 0) return fail(PKV_ERR_UNSUPPORTED, "num_kv_heads * head_dim not a multiple of 16");
  if (k_token_stride == 0) k_token_stride = row;
  if (v_token_stride == 0) v_token_stride = row;
  if (k_token_stride < row || v_token_stride < row)
    return fail(PKV_ERR_INVALID_ARG, "token stride smaller than num_kv_heads * head_dim");
  const int es = elem_bytes(dtype);
  if ((k_token_stride * es) % 16 != 0 || (v_token_stride * es) % 16 != 0)
    return fail(PKV_ERR_UNSUPPORTED, "token strides must be multiples of 16 bytes");
  if (num_tokens == 0) return PKV_OK;
  if (!k || !v || !slot_mapping || !k_cache || !v_cache) return fail(PKV_ERR_INVALID_ARG, "null pointer");
  if (!aligned16(k) || !aligned16(v) || !aligned16(k_cache) || !aligned16(v_cache))
    return fail(PKV_ERR_INVALID_ARG, "rows and caches must be 16-byte aligned");
  DeviceInfo* d = nullptr;
  pkv_status st = device_info(&d);
  if (st != PKV_OK) return st;
  cudaError_t e = launch_kv_write_fp8(k, v, slot_mapping, k_cache, v_cache, num_tokens, num_blocks * block_size,
                                      (int)row, es, k_token_stride, v_token_stride, k_scale, v_scale, d->err,
                                      static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "paged_kv_write_fp8 launch");
  return PKV_OK;
}

size_t paged_attention_workspace_size(int32_t num_seqs, int64_t num_tokens, int32_t num_q_heads,
                                      int32_t num_kv_heads, int32_t head_dim) {
  if (num_seqs < 0 || num_tokens < 0 || num_kv_heads <= 0 || num_q_heads <= 0 || head_dim <= 0) return 0;
  return workspace_layout(num_seqs, num_tokens, num_q_heads, num_kv_heads, head_dim, 0, 0, true).total;
}

size_t paged_attention_workspace_min(int32_t num_seqs, int64_t num_tokens, int32_t num_q_heads,
                                     int32_t num_kv_heads, int32_t head_dim) {
  if (num_seqs < 0 || num_tokens < 0 || num_kv_heads <= 0 || num_q_heads <= 0 || head_dim <= 0) return 0;
  return workspace_layout(num_seqs, num_tokens, num_q_heads, num_kv_heads, head_dim, 0, 0, false).total;
}

// The step's new K/V rows for a fused write (paged_kv_write_attention_forward):
// rows of row_dtype with token strides in elements (0: dense), copied (bf16 /
// f32 pools) or encoded as E4M3 codes (FP8 pools).
struct FusedWrite {
  const void* k;
  const void* v;
  const int64_t* slots;
  int64_t n, k_stride, v_stride;
  pkv_dtype row_dtype;
};

// Checks the fused write's arguments (as paged_kv_write / _fp8 do) and fills
// its stride defaults.
static pkv_status check_fused_write(FusedWrite* fw, int Hkv, int D, bool kv_fp8, pkv_dtype pool_dtype) {
  if (fw->n < 0) return fail(PKV_ERR_INVALID_ARG, "num_new_tokens must be >= 0");
  if (kv_fp8 ? (fw->row_dtype != PKV_DTYPE_BF16 && fw->row_dtype != PKV_DTYPE_F32) : fw->row_dtype != pool_dtype)
    return fail(PKV_ERR_UNSUPPORTED, "new rows of dtype %d for these pools", (int)fw->row_dtype);
  const int64_t row = (int64_t)Hkv * D;
  if (fw->k_stride == 0) fw->k_stride = row;
  if (fw->v_stride == 0) fw->v_stride = row;
  if (fw->k_stride < row || fw->v_stride < row)
    return fail(PKV_ERR_INVALID_ARG, "token stride smaller than num_kv_heads * head_dim");
  if (fw->n > 0 && (!fw->k || !fw->v || !fw->slots)) return fail(PKV_ERR_INVALID_ARG, "null pointer");
  if (kv_fp8) {
    const int es = elem_bytes(fw->row_dtype);
    if ((fw->k_stride * es) % 16 != 0 || (fw->v_stride * es) % 16 != 0 || !aligned16(fw->k) || !aligned16(fw->v))
      return fail(PKV_ERR_UNSUPPORTED, "new rows must be 16-byte aligned with strides of multiples of 16 bytes");
  }
  return PKV_OK;
}

// The forward call; kv_fp8: the pools hold E4M3 codes (q and out bf16), read
// as code * k_scale and code * v_scale.  fw: the step's new K/V rows, written
// first (by extra CTAs of the planner's launch where the rows allow it).
static pkv_status forward_impl(const void* q, const void* k_cache, const void* v_cache, const int32_t* block_tables,
                               const int32_t* context_lens, const int32_t* query_start_loc, void* out,
                               int32_t num_seqs, int64_t num_tokens, int32_t num_q_heads, int32_t num_kv_heads,
                               int32_t head_dim, int64_t num_blocks, int32_t block_size, int32_t max_blocks_per_seq,
                               int32_t max_query_len, float scale, int32_t causal, int32_t hints, void* workspace,
                               size_t workspace_bytes, pkv_dtype dtype, bool kv_fp8, float k_scale, float v_scale,
                               void* stream, const FusedWrite* fw = nullptr) {
  g_msg[0] = 0;
  const int B = num_seqs, Hq = num_q_heads, Hkv = num_kv_heads, D = head_dim, bs = block_size;
  const int64_t T = num_tokens;
  if (dtype != PKV_DTYPE_BF16 && dtype != PKV_DTYPE_F32) return fail(PKV_ERR_UNSUPPORTED, "dtype %d", (int)dtype);
  if (B < 0 || T < 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || num_blocks <= 0 || bs <= 0 || max_blocks_per_seq <= 0)
    return fail(PKV_ERR_INVALID_ARG, "sizes must be positive (num_seqs, num_tokens >= 0)");
  if (B > kMaxPlanSeqs) return fail(PKV_ERR_UNSUPPORTED, "more than %d sequences per call", kMaxPlanSeqs);
  if (Hq % Hkv != 0) return fail(PKV_ERR_INVALID_ARG, "num_q_heads (%d) %% num_kv_heads (%d) != 0", Hq, Hkv);
  if (Hq / Hkv > 128) return fail(PKV_ERR_UNSUPPORTED, "more than 128 q heads per kv head");
  if (D != 64 && D != 128) return fail(PKV_ERR_UNSUPPORTED, "head_dim %d (supported: 64, 128)", D);
  if (bs != 8 && bs != 16 && bs != 32 && bs != 64)
    return fail(PKV_ERR_UNSUPPORTED, "block_size %d (supported: 8, 16, 32, 64)", bs);
  if (!(scale > 0.f) || !isfinite(scale)) return fail(PKV_ERR_INVALID_ARG, "scale must be positive and finite");
  if ((int64_t)max_blocks_per_seq * bs > (int64_t)1 << 30) return fail(PKV_ERR_UNSUPPORTED, "context too long");
  if (T > ((int64_t)1 << 31) / ((int64_t)Hq * D)) return fail(PKV_ERR_UNSUPPORTED, "num_tokens too large");
  if (B == 0 || T == 0) {
    if (!fw || fw->n == 0) return PKV_OK;
    // nothing to attend: the write alone
    return kv_fp8 ? paged_kv_write_fp8(fw->k, fw->v, fw->slots, const_cast<void*>(k_cache),
                                       const_cast<void*>(v_cache), fw->n, num_blocks, bs, Hkv, D, fw->k_stride,
                                       fw->v_stride, fw->row_dtype, k_scale, v_scale, stream)
                  : paged_kv_write(fw->k, fw->v, fw->slots, const_cast<void*>(k_cache), const_cast<void*>(v_cache),
                                   fw->n, num_blocks, bs, Hkv, D, fw->k_stride, fw->v_stride, dtype, stream);
  }
  if (!q || !k_cache || !v_cache || !block_tables || !context_lens || !query_start_loc || !out)
    return fail(PKV_ERR_INVALID_ARG, "null pointer");
  if (!aligned16(q) || !aligned16(out) || !aligned16(k_cache) || !aligned16(v_cache))
    return fail(PKV_ERR_INVALID_ARG, "q, out and the caches must be 16-byte aligned");
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & (kAlign - 1)))
    return fail(PKV_ERR_WORKSPACE, "workspace missing or not 256-byte aligned");
  const WorkspaceLayout lay = workspace_layout(B, T, Hq, Hkv, D, workspace_bytes, 0, false);
  if (workspace_bytes < lay.total)
    return fail(PKV_ERR_WORKSPACE, "workspace of %zu bytes < minimum %zu", workspace_bytes, lay.total);

  DeviceInfo* dev = nullptr;
  pkv_status st = device_info(&dev);
  if (st != PKV_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const bool bf16 = dtype == PKV_DTYPE_BF16;
  const int G = Hq / Hkv;

  int dec_ctas = 1;
  cudaError_t e = kv_fp8 ? decode_fp8_ctas_per_sm(&dec_ctas) : decode_ctas_per_sm(bf16, D, &dec_ctas);
  if (e != cudaSuccess) return cuda_fail(e, "decode kernel set-up");

  uint8_t* ws = static_cast<uint8_t*>(workspace);
  PlanHeader* header = reinterpret_cast<PlanHeader*>(ws + lay.header_off);
  WorkItem* dec_items = reinterpret_cast<WorkItem*>(ws + lay.dec_off);
  WorkItem* mma_items = reinterpret_cast<WorkItem*>(ws + lay.mma_off);
  MergeGroup* merges = reinterpret_cast<MergeGroup*>(ws + lay.merge_off);
  int* tickets = reinterpret_cast<int*>(ws + lay.ticket_off);
  float2* part_ml = reinterpret_cast<float2*>(ws + lay.ml_off);
  float* part_acc = reinterpret_cast<float*>(ws + lay.acc_off);

  // tensor-core path for multi-token rows: bf16, head_dim 64 or 128, any G
  // up to 128 (an item is the floor(128 / G) whole tokens that fit 128 rows)
  const bool mma_ok = !kv_fp8 && bf16 && G <= kMmaRows;
  // decode-shaped rows: tensor-core kernel (keys on M, rows on N) for bf16,
  // head_dim 128 and G dividing 16; the CUDA-core kernel otherwise
  // FP8 pools: the same kernel on fp16 MMAs over converted tiles when the
  // host hint bounds every sequence's rows by 8, the CUDA-core kernel otherwise
  const bool f8tc = kv_fp8 && D == 128 && (G & (G - 1)) == 0 && max_query_len > 0 &&
                    (int64_t)max_query_len * G <= 8;
  const bool dectc = (mma_ok && D == 128 && (G & (G - 1)) == 0 && G <= kTcDecRows) || f8tc;
  const int dec_rows_max = dectc ? kTcDecRows : kDecRows;
  // rows of softmax per key in that kernel: a power of two >= G (so items hold
  // whole tokens) covering the hinted query length; 16 when there is no hint
  int tc_rows = kTcDecRows;
  if (dectc && max_query_len > 0) {
    const int64_t want = std::max<int64_t>(G, (int64_t)max_query_len * G);
    tc_rows = want <= 4 ? 4 : want <= 8 ? 8 : kTcDecRows;
  }
  // shared prefixes are read once per group by the tensor-core kernel, and
  // the rest of each member's keys by the tensor-core decode kernel
  const bool cascade = (hints & PKV_HINT_SHARED_PREFIX) != 0 && dectc && !kv_fp8;
  // with a host hint that no sequence has more rows than that, skip the launch
  const bool mma_launch =
      mma_ok && (cascade || !(max_query_len > 0 && (int64_t)max_query_len * G <= dec_rows_max));
  const int dec_grid = dev->sms * dec_ctas;

  PlanParams pp{};
  pp.context_lens = context_lens;
  pp.query_start_loc = query_start_loc;
  pp.B = B;
  pp.T = T;
  pp.G = G;
  pp.Hkv = Hkv;
  pp.bs = bs;
  pp.max_blocks = max_blocks_per_seq;
  pp.causal = causal ? 1 : 0;
  pp.mma_ok = mma_launch ? 1 : 0;
  pp.cascade = cascade ? 1 : 0;
  // The decode kernel runs beside the tensor-core kernel, on the SMs the plan
  // leaves it, unless it must read prefix partials that kernel writes.
  const bool side_by_side = mma_launch && dectc && !cascade;
  pp.side_by_side = side_by_side ? 1 : 0;
  pp.sms = dev->sms;
  const pkv_dtype kv_dtype = kv_fp8 ? PKV_DTYPE_FP8_E4M3 : dtype;
  pp.kv_key_bytes = 2 * D * elem_bytes(kv_dtype);
  pp.block_tables = block_tables;
  pp.dec_rows_max = dec_rows_max;
  pp.dec_unit_rows = dectc ? tc_rows : kDecRows;
  pp.mma_unit_rows = (kMmaRows / G) * G;
  pp.dec_tile_keys = dectc ? kMmaTileKeys : kDecTileKeys;
  // Four items per CTA of the decode kernels: fewer, longer items cost less
  // per item (pipeline restarts, partial writes, merges) than a finer tail
  // saves (measured on the decode, mixed and long-context batches).
  pp.target_dec = dectc ? dev->sms * 4 : dec_grid * 4;
  pp.dec_ctas = dectc ? dev->sms : dec_grid;
  // Items are fetched dynamically in largest-first order, so two per SM
  // balance the tensor-core kernel; every split costs a partial write and a
  // merge, so no more are made than that.
  pp.target_mma = dev->sms * 2;
  pp.min_chunk_dec = dectc ? 512 : 256;
  pp.min_chunk_mma = 512;
  pp.dec_cap = lay.dec_cap;
  pp.mma_cap = lay.mma_cap;
  pp.merge_cap = lay.merge_cap;
  pp.part_cap = lay.part_cap;
  pp.header = header;
  pp.dec_items = dec_items;
  pp.mma_items = mma_items;
  pp.merges = merges;
  pp.tickets = tickets;
  int* seq_scratch = reinterpret_cast<int*>(ws + lay.seq_off);
  pp.seq_pre = seq_scratch;
  pp.seq_grp = seq_scratch + B;
  pp.seq_mask = reinterpret_cast<uint32_t*>(seq_scratch + 2 * B);
  pp.seq_tmp = seq_scratch + 3 * B;
  pp.pre_groups = reinterpret_cast<PreGroup*>(ws + lay.pre_off);
  pp.out = out;
  pp.out_row_bytes = Hq * D * elem_bytes(dtype);
  pp.err = dev->err;
  if (fw && fw->n > 0) {
    // The new rows go in with the planner's launch when every row start is
    // 16-byte aligned (the vector copy, or the FP8 encoder); otherwise the
    // write kernel runs first, as paged_kv_write would.
    const int es = elem_bytes(fw->row_dtype);
    const int64_t row_bytes = (int64_t)Hkv * D * es;
    const bool vec = row_bytes % 16 == 0 && (fw->k_stride * es) % 16 == 0 && (fw->v_stride * es) % 16 == 0 &&
                     aligned16(fw->k) && aligned16(fw->v);
    if (vec) {
      pp.write_ctas = (int)std::min<int64_t>((fw->n + 15) / 16, 4 * (int64_t)dev->sms);
      pp.write_mode = kv_fp8 ? (fw->row_dtype == PKV_DTYPE_BF16 ? 2 : 3) : 1;
      pp.w_row = kv_fp8 ? Hkv * D : (int)(row_bytes / 16);
      pp.wk = fw->k;
      pp.wv = fw->v;
      pp.wslots = fw->slots;
      pp.wkc = const_cast<void*>(k_cache);
      pp.wvc = const_cast<void*>(v_cache);
      pp.wT = fw->n;
      pp.w_num_slots = num_blocks * bs;
      pp.wk_stride = kv_fp8 ? fw->k_stride : fw->k_stride * es;
      pp.wv_stride = kv_fp8 ? fw->v_stride : fw->v_stride * es;
      pp.wk_scale = k_scale;
      pp.wv_scale = v_scale;
    } else {
      e = launch_kv_write(fw->k, fw->v, fw->slots, const_cast<void*>(k_cache), const_cast<void*>(v_cache), fw->n,
                          num_blocks * bs, Hkv * D, es, fw->k_stride, fw->v_stride, dev->err, s);
      if (e != cudaSuccess) return cuda_fail(e, "paged_kv_write launch");
    }
  }
  if (cascade && (e = launch_prefix_search(pp, s)) != cudaSuccess) return cuda_fail(e, "prefix search launch");
  if ((e = launch_planner(pp, s)) != cudaSuccess) return cuda_fail(e, "planner launch");

  CUtensorMap kmap, vmap;
  if ((st = encode_pool_map(&kmap, k_cache, kv_dtype, num_blocks, bs, Hkv, D, D, CU_TENSOR_MAP_SWIZZLE_NONE)) !=
      PKV_OK)
    return st;
  if ((st = encode_pool_map(&vmap, v_cache, kv_dtype, num_blocks, bs, Hkv, D, D, CU_TENSOR_MAP_SWIZZLE_NONE)) !=
      PKV_OK)
    return st;

  AttnParams ap{};
  ap.q = q;
  ap.out = out;
  ap.block_tables = block_tables;
  ap.context_lens = context_lens;
  ap.query_start_loc = query_start_loc;
  ap.header = header;
  ap.part_ml = part_ml;
  ap.part_acc = part_acc;
  ap.groups = merges;
  ap.tickets = tickets;
  ap.Hq = Hq;
  ap.Hkv = Hkv;
  ap.G = G;
  ap.D = D;
  ap.bs = bs;
  ap.max_blocks = max_blocks_per_seq;
  ap.num_blocks = num_blocks;
  ap.scale_log2 = (kv_fp8 ? scale * k_scale : scale) * 1.4426950408889634f;
  ap.v_scale = kv_fp8 ? v_scale : 1.f;
  ap.causal = causal ? 1 : 0;
  ap.out_al32 = (reinterpret_cast<uintptr_t>(out) & 31u) == 0 ? 1 : 0;
  ap.mma_unit_rows = (kMmaRows / G) * G;
  ap.err = dev->err;
  ap.wait_ns = g_fault_wait_ns;
  ap.fault_tile = g_fault_tile;
  g_fault_tile = 0;
  g_fault_wait_ns = 0;

  // side by side: the decode kernel does not wait for the tensor-core grid,
  // and the tensor-core grid starts once the planner's grid has completed
  ap.no_wait = side_by_side ? 1 : 0;
  if (g_prof_start && (e = cudaEventRecord(g_prof_start, s)) != cudaSuccess) return cuda_fail(e, "profile event");
  if (mma_launch) {
    CUtensorMap qmap, kmap_sw, vmap_sw;
    if ((st = encode_q_map(&qmap, q, T, Hq, D, 64, G, kMmaRows / G)) != PKV_OK) return st;
    if ((st = encode_pool_map(&kmap_sw, k_cache, dtype, num_blocks, bs, Hkv, D, 64, CU_TENSOR_MAP_SWIZZLE_128B)) !=
        PKV_OK)
      return st;
    if ((st = encode_pool_map(&vmap_sw, v_cache, dtype, num_blocks, bs, Hkv, D, 64, CU_TENSOR_MAP_SWIZZLE_128B)) !=
        PKV_OK)
      return st;
    // the output in the q tile's layout: full 128-row tiles leave through TMA stores
    CUtensorMap omap;
    if ((st = encode_q_map(&omap, out, T, Hq, D, 64, G, kMmaRows / G)) != PKV_OK) return st;
    ap.counter = &header->mma_counter;
    ap.items = mma_items;
    if ((e = launch_mma(ap, qmap, kmap_sw, vmap_sw, omap, dev->sms, s)) != cudaSuccess)
      return cuda_fail(e, "mma launch");
  }
  if (g_prof_start && g_prof_mid && (e = cudaEventRecord(g_prof_mid, s)) != cudaSuccess)
    return cuda_fail(e, "profile event");
  ap.counter = &header->dec_counter;
  ap.items = dec_items;
  if (dectc && kv_fp8) {
    CUtensorMap qmap16;
    if ((st = encode_q_map(&qmap16, q, T, Hq, D, 64, G, kTcDecRows / G)) != PKV_OK) return st;
    // kmap / vmap (uint8, one {128, 1, bs, 1} box of codes per block) were encoded above
    if ((e = launch_dectc_fp8(ap, tc_rows, qmap16, kmap, vmap, dev->sms, s)) != cudaSuccess)
      return cuda_fail(e, "decode (tensor-core, FP8) launch");
  } else if (dectc) {
    CUtensorMap qmap16, kmap_sw, vmap_sw;
    if ((st = encode_q_map(&qmap16, q, T, Hq, D, 64, G, kTcDecRows / G)) != PKV_OK) return st;
    if ((st = encode_pool_map(&kmap_sw, k_cache, dtype, num_blocks, bs, Hkv, D, 64, CU_TENSOR_MAP_SWIZZLE_128B)) !=
        PKV_OK)
      return st;
    if ((st = encode_pool_map(&vmap_sw, v_cache, dtype, num_blocks, bs, Hkv, D, 64, CU_TENSOR_MAP_SWIZZLE_128B)) !=
        PKV_OK)
      return st;
    if ((e = launch_dectc(ap, tc_rows, qmap16, kmap_sw, vmap_sw, dev->sms, s)) != cudaSuccess)
      return cuda_fail(e, "decode (tensor-core) launch");
  } else if (kv_fp8) {
    if ((e = launch_decode_fp8(ap, kmap, vmap, dec_grid, s)) != cudaSuccess) return cuda_fail(e, "decode launch");
  } else if ((e = launch_decode(ap, kmap, vmap, bf16, dec_grid, s)) != cudaSuccess) {
    return cuda_fail(e, "decode launch");
  }
  if (g_prof_stop && (e = cudaEventRecord(g_prof_stop, s)) != cudaSuccess) return cuda_fail(e, "profile event");

  return PKV_OK;
}

pkv_status paged_attention_forward(const void* q, const void* k_cache, const void* v_cache,
                                   const int32_t* block_tables, const int32_t* context_lens,
                                   const int32_t* query_start_loc, void* out, int32_t num_seqs, int64_t num_tokens,
                                   int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim, int64_t num_blocks,
                                   int32_t block_size, int32_t max_blocks_per_seq, int32_t max_query_len,
                                   float scale, int32_t causal, int32_t hints, void* workspace,
                                   size_t workspace_bytes, pkv_dtype dtype, void* stream) {
  return forward_impl(q, k_cache, v_cache, block_tables, context_lens, query_start_loc, out, num_seqs, num_tokens,
                      num_q_heads, num_kv_heads, head_dim, num_blocks, block_size, max_blocks_per_seq, max_query_len,
                      scale, causal, hints, workspace, workspace_bytes, dtype, false, 1.f, 1.f, stream);
}

pkv_status paged_kv_write_attention_forward(const void* k, const void* v, const int64_t* slot_mapping,
                                            int64_t num_new_tokens, int64_t k_token_stride, int64_t v_token_stride,
                                            const void* q, const void* k_cache, const void* v_cache,
                                            const int32_t* block_tables, const int32_t* context_lens,
                                            const int32_t* query_start_loc, void* out, int32_t num_seqs,
                                            int64_t num_tokens, int32_t num_q_heads, int32_t num_kv_heads,
                                            int32_t head_dim, int64_t num_blocks, int32_t block_size,
                                            int32_t max_blocks_per_seq, int32_t max_query_len, float scale,
                                            int32_t causal, int32_t hints, void* workspace, size_t workspace_bytes,
                                            pkv_dtype dtype, void* stream) {
  g_msg[0] = 0;
  FusedWrite fw{k, v, slot_mapping, num_new_tokens, k_token_stride, v_token_stride, dtype};
  if (num_kv_heads <= 0 || head_dim <= 0) return fail(PKV_ERR_INVALID_ARG, "sizes must be positive");
  pkv_status st = check_fused_write(&fw, num_kv_heads, head_dim, false, dtype);
  if (st != PKV_OK) return st;
  return forward_impl(q, k_cache, v_cache, block_tables, context_lens, query_start_loc, out, num_seqs, num_tokens,
                      num_q_heads, num_kv_heads, head_dim, num_blocks, block_size, max_blocks_per_seq, max_query_len,
                      scale, causal, hints, workspace, workspace_bytes, dtype, false, 1.f, 1.f, stream, &fw);
}

pkv_status paged_kv_write_attention_forward_fp8kv(
    const void* k, const void* v, const int64_t* slot_mapping, int64_t num_new_tokens, int64_t k_token_stride,
    int64_t v_token_stride, pkv_dtype row_dtype, const void* q, const void* k_cache, const void* v_cache,
    const int32_t* block_tables, const int32_t* context_lens, const int32_t* query_start_loc, void* out,
    int32_t num_seqs, int64_t num_tokens, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
    int64_t num_blocks, int32_t block_size, int32_t max_blocks_per_seq, int32_t max_query_len, float scale,
    int32_t causal, float k_scale, float v_scale, int32_t hints, void* workspace, size_t workspace_bytes,
    void* stream) {
  g_msg[0] = 0;
  if (!(k_scale > 0.f) || !isfinite(k_scale) || !(v_scale > 0.f) || !isfinite(v_scale))
    return fail(PKV_ERR_INVALID_ARG, "k_scale and v_scale must be positive and finite");
  if (head_dim != 128) return fail(PKV_ERR_UNSUPPORTED, "head_dim %d with an FP8 cache (supported: 128)", head_dim);
  if (num_kv_heads <= 0) return fail(PKV_ERR_INVALID_ARG, "sizes must be positive");
  FusedWrite fw{k, v, slot_mapping, num_new_tokens, k_token_stride, v_token_stride, row_dtype};
  pkv_status st = check_fused_write(&fw, num_kv_heads, head_dim, true, PKV_DTYPE_FP8_E4M3);
  if (st != PKV_OK) return st;
  return forward_impl(q, k_cache, v_cache, block_tables, context_lens, query_start_loc, out, num_seqs, num_tokens,
                      num_q_heads, num_kv_heads, head_dim, num_blocks, block_size, max_blocks_per_seq, max_query_len,
                      scale, causal, hints, workspace, workspace_bytes, PKV_DTYPE_BF16, true, k_scale, v_scale,
                      stream, &fw);
}

pkv_status paged_attention_forward_fp8kv(const void* q, const void* k_cache, const void* v_cache,
                                         const int32_t* block_tables, const int32_t* context_lens,
                                         const int32_t* query_start_loc, void* out, int32_t num_seqs,
                                         int64_t num_tokens, int32_t num_q_heads, int32_t num_kv_heads,
                                         int32_t head_dim, int64_t num_blocks, int32_t block_size,
                                         int32_t max_blocks_per_seq, int32_t max_query_len, float scale,
                                         int32_t causal, float k_scale, float v_scale, int32_t hints,
                                         void* workspace, size_t workspace_bytes, void* stream) {
  g_msg[0] = 0;
  if (!(k_scale > 0.f) || !isfinite(k_scale) || !(v_scale > 0.f) || !isfinite(v_scale))
    return fail(PKV_ERR_INVALID_ARG, "k_scale and v_scale must be positive and finite");
  if (head_dim != 128) return fail(PKV_ERR_UNSUPPORTED, "head_dim %d with an FP8 cache (supported: 128)", head_dim);
  return forward_impl(q, k_cache, v_cache, block_tables, context_lens, query_start_loc, out, num_seqs, num_tokens,
                      num_q_heads, num_kv_heads, head_dim, num_blocks, block_size, max_blocks_per_seq, max_query_len,
                      scale, causal, hints, workspace, workspace_bytes, PKV_DTYPE_BF16, true, k_scale, v_scale,
                      stream);
}

}  // extern "C"
