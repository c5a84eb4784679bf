// Slot-mapping scatter of new K/V rows into the block pool.
//
// "ADR 004: Paged Attention Serving Integration", Decision 4: the model
// writes K/V into the block allocator; "Paged Attention 基础", section 2:
// token position -> (physical block, slot).  Slot s addresses pool row
// s = block * block_size + offset, and a pool row is the contiguous
// num_kv_heads * head_dim elements of one token, so the write is a gather-free
// row copy: read the token's row (contiguous, or with a token stride) and
// store it at row s of k_cache / v_cache.
//
// HBM-bound: one warp per token, 16-byte vector loads (read-only, no L1
// allocation) and stores, all of a token's K and V chunks in flight before
// the first store.
#include "kv_rows.cuh"
#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace {

// Vector path: every row start is 16-byte aligned and a row is a multiple of
// 16 bytes.  kChunks = chunks per lane held in registers per pass.
template <int kChunks>
__global__ void __launch_bounds__(256) kv_write_vec(const uint8_t* __restrict__ k, const uint8_t* __restrict__ v,
                                                    const int64_t* __restrict__ slots, uint8_t* kc, uint8_t* vc,
                                                    int64_t T, int64_t num_slots, int row_chunks,
                                                    int64_t k_stride_b, int64_t v_stride_b, int* err) {
  pdl_launch_dependents();  // a following planner reads nothing this kernel writes
  const int lane = threadIdx.x & 31;
  const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
  for (int64_t t = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; t < T; t += warps)
    copy_token_rows<kChunks>(k, v, slots, kc, vc, t, num_slots, row_chunks, k_stride_b, v_stride_b, err, lane);
}

// Element path for rows that are not 16-byte aligned (odd strides): one warp
// per token copying `unit`-byte elements.
template <typename U>
__global__ void __launch_bounds__(256) kv_write_elem(const U* __restrict__ k, const U* __restrict__ v,
                                                     const int64_t* __restrict__ slots, U* kc, U* vc, int64_t T,
                                                     int64_t num_slots, int row_elems, int64_t k_stride,
                                                     int64_t v_stride, int* err) {
  const int lane = threadIdx.x & 31;
  const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
  for (int64_t t = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; t < T; t += warps) {
    const int64_t s = slots[t];
    if (s < 0) continue;
    if (s >= num_slots) {
      if (lane == 0) raise_error(err, PKV_DEVERR_SLOT_OUT_OF_RANGE);
      continue;
    }
    for (int e = lane; e < row_elems; e += 32) {
      kc[s * row_elems + e] = k[t * k_stride + e];
      vc[s * row_elems + e] = v[t * v_stride + e];
    }
  }
}

// FP8 (E4M3) cache write: one warp per token (quantize_token_rows).
template <typename U>
__global__ void __launch_bounds__(256) kv_write_fp8_kernel(const U* __restrict__ k, const U* __restrict__ v,
                                                           const int64_t* __restrict__ slots, uint8_t* kc,
                                                           uint8_t* vc, int64_t T, int64_t num_slots, int row_elems,
                                                           int64_t k_stride, int64_t v_stride, float k_scale,
                                                           float v_scale, int* err) {
  pdl_launch_dependents();  // a following planner reads nothing this kernel writes
  const int lane = threadIdx.x & 31;
  const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
  for (int64_t t = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; t < T; t += warps)
    quantize_token_rows<U>(k, v, slots, kc, vc, t, num_slots, row_elems, k_stride, v_stride, k_scale, v_scale, err,
                           lane);
}

}  // namespace

cudaError_t launch_kv_write_fp8(const void* k, const void* v, const int64_t* slots, void* kc, void* vc, int64_t T,
                                int64_t num_slots, int row_elems, int es, int64_t k_stride, int64_t v_stride,
                                float k_scale, float v_scale, int* err, cudaStream_t s) {
  if (T <= 0) return cudaSuccess;
  const int64_t blocks64 = (T + 7) / 8;
  const int blocks = (int)(blocks64 < 65535 * 8 ? blocks64 : 65535 * 8);
  if (es == 2) {
    kv_write_fp8_kernel<uint16_t><<<blocks, 256, 0, s>>>((const uint16_t*)k, (const uint16_t*)v, slots, (uint8_t*)kc,
                                                          (uint8_t*)vc, T, num_slots, row_elems, k_stride, v_stride,
                                                          k_scale, v_scale, err);
  } else {
    kv_write_fp8_kernel<float><<<blocks, 256, 0, s>>>((const float*)k, (const float*)v, slots, (uint8_t*)kc,
                                                       (uint8_t*)vc, T, num_slots, row_elems, k_stride, v_stride,
                                                       k_scale, v_scale, err);
  }
  return cudaGetLastError();
}

cudaError_t launch_kv_write(const void* k, const void* v, const int64_t* slots, void* kc, void* vc, int64_t T,
                            int64_t num_slots, int row_elems, int elem_bytes, int64_t k_stride, int64_t v_stride,
                            int* err, cudaStream_t s) {
  if (T <= 0) return cudaSuccess;
  const int64_t row_bytes = (int64_t)row_elems * elem_bytes;
  const bool aligned = (row_bytes % 16 == 0) && ((k_stride * elem_bytes) % 16 == 0) &&
                       ((v_stride * elem_bytes) % 16 == 0) && (reinterpret_cast<uintptr_t>(k) % 16 == 0) &&
                       (reinterpret_cast<uintptr_t>(v) % 16 == 0) && (reinterpret_cast<uintptr_t>(kc) % 16 == 0) &&
                       (reinterpret_cast<uintptr_t>(vc) % 16 == 0);
  const int threads = 256;
  const int64_t blocks64 = (T + 7) / 8;
  const int blocks = (int)(blocks64 < 65535 * 8 ? blocks64 : 65535 * 8);
  if (aligned) {
    const int chunks = (int)(row_bytes / 16);
    if (chunks <= 32 * 2) {
      kv_write_vec<2><<<blocks, threads, 0, s>>>((const uint8_t*)k, (const uint8_t*)v, slots, (uint8_t*)kc,
                                                  (uint8_t*)vc, T, num_slots, chunks, k_stride * elem_bytes,
                                                  v_stride * elem_bytes, err);
    } else {
      kv_write_vec<4><<<blocks, threads, 0, s>>>((const uint8_t*)k, (const uint8_t*)v, slots, (uint8_t*)kc,
                                                  (uint8_t*)vc, T, num_slots, chunks, k_stride * elem_bytes,
                                                  v_stride * elem_bytes, err);
    }
  } else if (elem_bytes == 4) {
    kv_write_elem<uint32_t><<<blocks, threads, 0, s>>>((const uint32_t*)k, (const uint32_t*)v, slots,
                                                        (uint32_t*)kc, (uint32_t*)vc, T, num_slots, row_elems,
                                                        k_stride, v_stride, err);
  } else {
    kv_write_elem<uint16_t><<<blocks, threads, 0, s>>>((const uint16_t*)k, (const uint16_t*)v, slots,
                                                        (uint16_t*)kc, (uint16_t*)vc, T, num_slots, row_elems,
                                                        k_stride, v_stride, err);
  }
  return cudaGetLastError();
}

}  // namespace pkv
