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

}  // namespace

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
