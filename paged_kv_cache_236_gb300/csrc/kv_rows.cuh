// One token's slot-mapping scatter, as one warp does it: the device routines
// shared by the K/V write kernels and by the extra CTAs of the planner's
// grid that write a step's new rows in the same launch.
//
// "ADR 004: Paged Attention Serving Integration", Decision 4: the model
// writes K/V into the block allocator; "Paged Attention 基础", section 2:
// token position -> (physical block, slot).  Slot s addresses pool row s =
// block * block_size + offset; a pool row is the contiguous
// num_kv_heads * head_dim elements of one token, so the write is a row copy.
#pragma once

#include <cuda_fp8.h>

#include "pkv_device.cuh"

namespace pkv {

__device__ __forceinline__ int4 ld_stream(const int4* p) {
  int4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.s32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

// Copy token t's K and V rows (row_chunks 16-byte chunks each; every row
// start 16-byte aligned) to pool row slots[t] of kc / vc.  The whole warp
// calls it; all of a pass's loads are in flight before its stores.  Slots
// < 0 are skipped; slots >= num_slots are skipped and flagged.
template <int kChunks>
__device__ __forceinline__ void copy_token_rows(const uint8_t* __restrict__ k, const uint8_t* __restrict__ v,
                                                const int64_t* __restrict__ slots, uint8_t* kc, uint8_t* vc,
                                                int64_t t, int64_t num_slots, int row_chunks, int64_t k_stride_b,
                                                int64_t v_stride_b, int* err, int lane) {
  const int64_t s = slots[t];
  if (s < 0) return;
  if (s >= num_slots) {
    if (lane == 0) raise_error(err, PKV_DEVERR_SLOT_OUT_OF_RANGE);
    return;
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

// The FP8 (E4M3) cache write of token t: code = e4m3(RNE(x / scale)),
// saturating at +-448 (the division is IEEE fp32); U is the row element
// (uint16_t: bf16 bits, float: fp32).  16 elements a lane per pass: one
// 16-byte store of codes from 32 (bf16) or 64 (fp32) bytes of row.  Row
// starts and strides are multiples of 16 bytes.
template <typename U>
__device__ __forceinline__ void quantize_token_rows(const U* __restrict__ k, const U* __restrict__ v,
                                                    const int64_t* __restrict__ slots, uint8_t* kc, uint8_t* vc,
                                                    int64_t t, int64_t num_slots, int row_elems, int64_t k_stride,
                                                    int64_t v_stride, float k_scale, float v_scale, int* err,
                                                    int lane) {
  const int64_t s = slots[t];
  if (s < 0) return;
  if (s >= num_slots) {
    if (lane == 0) raise_error(err, PKV_DEVERR_SLOT_OUT_OF_RANGE);
    return;
  }
  constexpr int kVec = 16 / sizeof(U);  // elements per 16-byte load
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
        const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(__fdiv_rn(x[4 * i], sc), __fdiv_rn(x[4 * i + 1], sc)),
                                                     __NV_SATFINITE, __NV_E4M3);
        const uint32_t hi = __nv_cvt_float2_to_fp8x2(
            make_float2(__fdiv_rn(x[4 * i + 2], sc), __fdiv_rn(x[4 * i + 3], sc)), __NV_SATFINITE, __NV_E4M3);
        out[i] = (lo & 0xFFFFu) | (hi << 16);
      }
      uint8_t* dst = (which ? vc : kc) + s * row_elems + e0;
      *reinterpret_cast<uint4*>(dst) = make_uint4(out[0], out[1], out[2], out[3]);
    }
  }
}

}  // namespace pkv
