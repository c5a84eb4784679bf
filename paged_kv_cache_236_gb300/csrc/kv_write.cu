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
#include <cuda_fp8.h>

#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace {

__device__ __forceinline__ int4 ld_stream(const int4* p) {
  int4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.s32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

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
  for (int64_t t = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; t < T; t += warps) {
    const int64_t s = slots[t];
    if (s < 0) continue;
    if (s >= num_slots) {
      if (lane == 0) raise_error(err, PKV_DEVERR_SLOT_OUT_OF_RANGE);
      continue;
    }
    const int4* ks = reinterpret_cast<const int4*>(k + t * k_stride_b);
    const int4* vs = reinterpret_cast<const int4*>(v + t * v_stride_b);
    int4* kd = reinterpret_cast<int4*>(kc + s * (int64_t)row_chunks * 16);
    int4* vd = reinterpret_cast<int4*>(vc + s * (int64_t)row_chunks * 16);
    for (int base = 0; base < row_chunks; base += 32 * kChunks) {
      int4 kr[kChunks], vr[kChunks];
#pragma unroll
      for (int i = 0; i < kChunks; ++i) {
        const int c = base + i * 32 + lane;
        if (c < row_chunks) {
          kr[i] = ld_stream(ks + c);
          vr[i] = ld_stream(vs + c);
        }
      }
#pragma unroll
      for (int i = 0; i < kChunks; ++i) {
        const int c = base + i * 32 + lane;
        if (c < row_chunks) {
          kd[c] = kr[i];
          vd[c] = vr[i];
        }
      }
    }
  }
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

// FP8 (E4M3) cache write: code = e4m3(RNE(x / scale)), saturating at +-448
// (the division is IEEE fp32).  One warp per token, 16 elements a lane per
// pass: one 16-byte store of codes from 32 (bf16) or 64 (fp32) bytes of row.
template <typename U>
__global__ void __launch_bounds__(256) kv_write_fp8_kernel(const U* __restrict__ k, const U* __restrict__ v,
                                                           const int64_t* __restrict__ slots, uint8_t* kc,
                                                           uint8_t* vc, int64_t T, int64_t num_slots, int row_elems,
                                                           int64_t k_stride, int64_t v_stride, float k_scale,
                                                           float v_scale, int* err) {
  pdl_launch_dependents();  // a following planner reads nothing this kernel writes
  const int lane = threadIdx.x & 31;
  const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
  constexpr int kVec = 16 / sizeof(U);  // elements per 16-byte load
  for (int64_t t = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; t < T; t += warps) {
    const int64_t s = slots[t];
    if (s < 0) continue;
    if (s >= num_slots) {
      if (lane == 0) raise_error(err, PKV_DEVERR_SLOT_OUT_OF_RANGE);
      continue;
    }
    for (int e0 = lane * 16; e0 < row_elems; e0 += 32 * 16) {
#pragma unroll
      for (int which = 0; which < 2; ++which) {
        const U* src = (which ? v + t * v_stride : k + t * k_stride) + e0;
        const float sc = which ? v_scale : k_scale;
        float x[16];
#pragma unroll
        for (int c = 0; c < 16 / kVec; ++c) {
          const int4 r = ld_stream(reinterpret_cast<const int4*>(src) + c);
          const uint32_t w[4] = {(uint32_t)r.x, (uint32_t)r.y, (uint32_t)r.z, (uint32_t)r.w};
          if constexpr (sizeof(U) == 2) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              x[c * 8 + 2 * i] = __uint_as_float(w[i] << 16);
              x[c * 8 + 2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
            }
          } else {
#pragma unroll
            for (int i = 0; i < 4; ++i) x[c * 4 + i] = __uint_as_float(w[i]);
          }
        }
        uint32_t out[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const uint32_t lo = __nv_cvt_float2_to_fp8x2(
              make_float2(__fdiv_rn(x[4 * i], sc), __fdiv_rn(x[4 * i + 1], sc)), __NV_SATFINITE, __NV_E4M3);
          const uint32_t hi = __nv_cvt_float2_to_fp8x2(
              make_float2(__fdiv_rn(x[4 * i + 2], sc), __fdiv_rn(x[4 * i + 3], sc)), __NV_SATFINITE, __NV_E4M3);
          out[i] = (lo & 0xFFFFu) | (hi << 16);
        }
        uint8_t* dst = (which ? vc : kc) + s * row_elems + e0;
        *reinterpret_cast<uint4*>(dst) = make_uint4(out[0], out[1], out[2], out[3]);
      }
    }
  }
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
