// CUDA-core paged attention for few rows per kv head (decode), with split-KV,
// plus the split merge.
//
// What it computes ("Paged Attention 基础", section 2, steps 1-5): for each
// work item - up to kDecRows rows (query token, head-in-group) of one
// sequence and one kv head, over keys [kb, ke) - walk the block table, fetch
// each key block, form scale * q.k, apply the causal mask at the query's
// absolute position L - n + i, and accumulate softmax(.)V with a running
// (max, sum) ("online softmax").  Items that cover a whole key range write
// normalised output rows; split items write partial (m, l, acc) rows that
// merge_kernel combines: m = max_p m_p, l = sum_p l_p 2^(m_p - m),
// O = sum_p acc_p 2^(m_p - m) / l (logits kept in log2 units).
//
// GB300 design:
//  * persistent CTAs (2 per SM) fetch items from an atomic counter;
//  * a producer warp streams each 64-key tile of K and V with TMA: one 4-D
//    tensor-map box per physical block ({head_dim, 1 head, block_size, 1
//    block} of the pool [num_blocks, block_size, num_kv_heads, head_dim]), so
//    the block table is resolved by the box coordinate and blocks past a
//    sequence's end (or invalid ids) are out-of-range boxes that read as
//    zeros; a 3-stage mbarrier ring keeps ~64 KB per CTA in flight;
//  * 4 consumer warps each own 16 keys of a tile: 8 lanes per key (16-byte
//    shared loads, conflict-free), partial dot products for the 4 rows of 2
//    keys reduced with a transposing butterfly (7 shuffles per 8 scores),
//    warp-level online softmax, then P.V with each lane owning head_dim/32
//    output columns of all 4 rows; the 4 warp states are merged at the end of
//    an item through shared memory.
#include <math_constants.h>

#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace {

constexpr int kConsumerWarps = 4;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kWarpKeys = kDecTileKeys / kConsumerWarps;  // 16
constexpr int kRP = kDecRows;                             // 4 rows per item
constexpr int kLPT = 8;                                   // lanes per key (QK)
constexpr int kTPR = kLPT / kRP;                          // keys per lane group per round (2)
constexpr int kKeysPerRound = (32 / kLPT) * kTPR;         // 8
constexpr int kRounds = kWarpKeys / kKeysPerRound;        // 2
constexpr int kMetaDone = 2, kMetaLast = 1;
static_assert(kRP == 4 && kLPT == 8, "butterfly below is written for 8 partials per lane");

template <typename T, int D>
struct Cfg {
  static constexpr int kEs = sizeof(T);
  static constexpr int kRowBytes = D * kEs;
  static constexpr int kChunks = kRowBytes / 16;
  static constexpr int kCPL = kChunks / kLPT;  // 16-byte chunks per lane per key
  static constexpr int kEPC = 16 / kEs;        // elements per chunk
  static constexpr int kEPL = kCPL * kEPC;     // q elements per lane
  static constexpr int kDPL = D / 32;          // output columns per lane
  static constexpr int kTileBytes = kDecTileKeys * kRowBytes;
  static constexpr int kStageBytes = 2 * kTileBytes;
  static constexpr int kStages = (98304 / kStageBytes) < 2 ? 2 : ((98304 / kStageBytes) > 4 ? 4 : (98304 / kStageBytes));
  // shared memory carve-up
  static constexpr int kPOff = kStages * kStageBytes;
  static constexpr int kPBytes = kConsumerWarps * kWarpKeys * kRP * 4;
  static constexpr int kAccOff = kPOff + kPBytes;
  static constexpr int kAccBytes = kConsumerWarps * kRP * D * 4;
  static constexpr int kMlOff = kAccOff + kAccBytes;
  static constexpr int kMlBytes = kConsumerWarps * kRP * 2 * 4;
  static constexpr int kMetaOff = kMlOff + kMlBytes;
  static constexpr int kMetaBytes = kStages * 16;
  static constexpr int kBarOff = kMetaOff + kMetaBytes;
  static constexpr int kSmem = kBarOff + 2 * kStages * 8 + 1024;  // + slack to align the base to 1 KB
  static_assert(kCPL >= 1 && kChunks % kLPT == 0, "row must split into 8 lanes of 16-byte chunks");
};

struct alignas(16) Meta {
  int item, kbase, flags, pad;
};

template <int kBytes>
struct VecT;
template <>
struct VecT<4> {
  using type = uint32_t;
};
template <>
struct VecT<8> {
  using type = uint2;
};
template <>
struct VecT<16> {
  using type = uint4;
};

// Convert one 16-byte chunk of K into floats.
template <typename T>
__device__ __forceinline__ void chunk_to_float(const uint4 raw, float* f);
template <>
__device__ __forceinline__ void chunk_to_float<__nv_bfloat16>(const uint4 raw, float* f) {
  f[0] = bf16_lo(raw.x);
  f[1] = bf16_hi(raw.x);
  f[2] = bf16_lo(raw.y);
  f[3] = bf16_hi(raw.y);
  f[4] = bf16_lo(raw.z);
  f[5] = bf16_hi(raw.z);
  f[6] = bf16_lo(raw.w);
  f[7] = bf16_hi(raw.w);
}
template <>
__device__ __forceinline__ void chunk_to_float<float>(const uint4 raw, float* f) {
  f[0] = __uint_as_float(raw.x);
  f[1] = __uint_as_float(raw.y);
  f[2] = __uint_as_float(raw.z);
  f[3] = __uint_as_float(raw.w);
}

// Load this lane's kDPL V columns of one key row as floats.
template <typename T, int DPL>
__device__ __forceinline__ void load_v(const uint8_t* p, float* f) {
  if constexpr (sizeof(T) == 2) {
    if constexpr (DPL == 4) {
      const uint2 w = *reinterpret_cast<const uint2*>(p);
      f[0] = bf16_lo(w.x);
      f[1] = bf16_hi(w.x);
      f[2] = bf16_lo(w.y);
      f[3] = bf16_hi(w.y);
    } else {
      const uint32_t w = *reinterpret_cast<const uint32_t*>(p);
      f[0] = bf16_lo(w);
      f[1] = bf16_hi(w);
    }
  } else {
    if constexpr (DPL == 4) {
      const float4 w = *reinterpret_cast<const float4*>(p);
      f[0] = w.x;
      f[1] = w.y;
      f[2] = w.z;
      f[3] = w.w;
    } else {
      const float2 w = *reinterpret_cast<const float2*>(p);
      f[0] = w.x;
      f[1] = w.y;
    }
  }
}

// Sum v[i] over the 8 lanes of a lane group, transposing: afterwards lane
// (lane & 7) == i holds the group total of v[i] in v[0].
__device__ __forceinline__ float group_transpose_sum(float v[8], int lane) {
  const bool b2 = lane & 4, b1 = lane & 2, b0 = lane & 1;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float send = b2 ? v[i] : v[i + 4];
    const float keep = b2 ? v[i + 4] : v[i];
    v[i] = keep + __shfl_xor_sync(0xffffffffu, send, 4);
  }
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const float send = b1 ? v[i] : v[i + 2];
    const float keep = b1 ? v[i + 2] : v[i];
    v[i] = keep + __shfl_xor_sync(0xffffffffu, send, 2);
  }
  const float send = b0 ? v[0] : v[1];
  const float keep = b0 ? v[1] : v[0];
  return keep + __shfl_xor_sync(0xffffffffu, send, 1);
}

template <typename T, int D>
__global__ void __launch_bounds__(kThreads, 2) decode_kernel(const AttnParams p,
                                                             const __grid_constant__ CUtensorMap kmap,
                                                             const __grid_constant__ CUtensorMap vmap) {
  using C = Cfg<T, D>;
  extern __shared__ __align__(16) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  float* pbuf = reinterpret_cast<float*>(smem + C::kPOff);
  float* comb_acc = reinterpret_cast<float*>(smem + C::kAccOff);
  float* comb_ml = reinterpret_cast<float*>(smem + C::kMlOff);
  Meta* meta = reinterpret_cast<Meta*>(smem + C::kMetaOff);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::kBarOff);
  uint64_t* empty = full + C::kStages;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_items = p.header->n_dec;
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kConsumerWarps);
    }
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == kConsumerWarps) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tensormap(&kmap);
      prefetch_tensormap(&vmap);
    }
    const int nb_per_tile = kDecTileKeys / p.bs;
    int tile = 0;
    for (;;) {
      int idx = 0;
      if (lane == 0) idx = atomicAdd(p.counter, 1);
      idx = __shfl_sync(0xffffffffu, idx, 0);
      const int stage0 = tile % C::kStages;
      if (idx >= n_items) {
        if (!mbar_wait(&empty[stage0], ((tile / C::kStages) & 1) ^ 1, p.err)) return;
        if (lane == 0) {
          meta[stage0].item = -1;
          meta[stage0].flags = kMetaDone;
          mbar_arrive(&full[stage0]);
        }
        break;
      }
      const WorkItem it = p.items[idx];
      const int L = p.context_lens[it.seq];
      const int nblk = (L + p.bs - 1) / p.bs;
      const int32_t* bt = p.block_tables + (int64_t)it.seq * p.max_blocks;
      for (int kbase = it.kb; kbase < it.ke; kbase += kDecTileKeys) {
        const int stage = tile % C::kStages;
        if (!mbar_wait(&empty[stage], ((tile / C::kStages) & 1) ^ 1, p.err)) return;
        if (lane == 0) {
          meta[stage].item = idx;
          meta[stage].kbase = kbase;
          meta[stage].flags = (kbase + kDecTileKeys >= it.ke) ? kMetaLast : 0;
          mbar_arrive_expect_tx(&full[stage], C::kStageBytes);
        }
        __syncwarp();
        if (lane < nb_per_tile) {
          const int lb = kbase / p.bs + lane;
          int phys = (int)p.num_blocks;  // out of range: the box reads as zeros
          if (lb < nblk) {
            const int b = bt[lb];
            if (b >= 0 && (int64_t)b < p.num_blocks)
              phys = b;
            else
              raise_error(p.err, PKV_DEVERR_BLOCK_OUT_OF_RANGE);
          }
          uint8_t* kdst = smem + stage * C::kStageBytes + lane * p.bs * C::kRowBytes;
          tma_load_4d(kdst, &kmap, &full[stage], 0, it.kvh, 0, phys);
          tma_load_4d(kdst + C::kTileBytes, &vmap, &full[stage], 0, it.kvh, 0, phys);
        }
        ++tile;
      }
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const int grp = lane >> 3, j = lane & 7;
  const int myrow = lane & (kRP - 1);  // row whose scores this lane holds
  float* pw = pbuf + warp * kWarpKeys * kRP;

  float qf[kRP][C::kEPL];
  float acc[kRP][C::kDPL];
  float m_row = -CUDART_INF_F, l_row = 0.f;
  int vis_row = 0;  // keys visible to row `myrow` (absolute key < vis_row)
  WorkItem it = {0, 0, 0, 0, 0, 0, -1, 0};
  int L = 0, n = 0, qstart = 0;
  int cur = -1;
  int tile = 0;
  for (;;) {
    const int stage = tile % C::kStages;
    if (!mbar_wait(&full[stage], (tile / C::kStages) & 1, p.err)) break;
    const Meta mt = meta[stage];
    if (mt.flags & kMetaDone) break;
    if (mt.item != cur) {
      cur = mt.item;
      it = p.items[cur];
      L = p.context_lens[it.seq];
      qstart = p.query_start_loc[it.seq];
      n = p.query_start_loc[it.seq + 1] - qstart;
      m_row = -CUDART_INF_F;
      l_row = 0.f;
#pragma unroll
      for (int r = 0; r < kRP; ++r) {
#pragma unroll
        for (int e = 0; e < C::kDPL; ++e) acc[r][e] = 0.f;
        const int row = it.row0 + r;
        if (r < it.nrows) {
          const int tok = row / p.G, g = row - tok * p.G;
          const T* qrow = reinterpret_cast<const T*>(p.q) +
                          ((int64_t)(qstart + tok) * p.Hq + (int64_t)it.kvh * p.G + g) * D;
#pragma unroll
          for (int m = 0; m < C::kCPL; ++m) {
            const uint4 raw = *reinterpret_cast<const uint4*>(qrow + (j + 8 * m) * C::kEPC);
            float f[C::kEPC];
            chunk_to_float<T>(raw, f);
#pragma unroll
            for (int e = 0; e < C::kEPC; ++e) qf[r][m * C::kEPC + e] = f[e] * p.scale_log2;
          }
        } else {
#pragma unroll
          for (int e = 0; e < C::kEPL; ++e) qf[r][e] = 0.f;
        }
      }
      {
        const int row = it.row0 + myrow;
        const int tok = row / p.G;
        vis_row = myrow < it.nrows ? min(it.ke, p.causal ? L - n + tok + 1 : L) : 0;
      }
    }
    const uint8_t* ks = smem + stage * C::kStageBytes + warp * kWarpKeys * C::kRowBytes;
    const uint8_t* vs = ks + C::kTileBytes;
    const int wkb = mt.kbase + warp * kWarpKeys;  // absolute key of this warp's first key

    // ---- scores: s = (scale*log2e) q.k for 4 rows x 16 keys, 2 per lane
    float sc[kRounds];
#pragma unroll
    for (int rnd = 0; rnd < kRounds; ++rnd) {
      float part[kTPR * kRP];
#pragma unroll
      for (int i = 0; i < kTPR * kRP; ++i) part[i] = 0.f;
#pragma unroll
      for (int t = 0; t < kTPR; ++t) {
        const int kl = rnd * kKeysPerRound + grp * kTPR + t;
        const uint8_t* krow = ks + kl * C::kRowBytes;
#pragma unroll
        for (int m = 0; m < C::kCPL; ++m) {
          const uint4 raw = *reinterpret_cast<const uint4*>(krow + (j + 8 * m) * 16);
          float f[C::kEPC];
          chunk_to_float<T>(raw, f);
#pragma unroll
          for (int r = 0; r < kRP; ++r)
#pragma unroll
            for (int e = 0; e < C::kEPC; ++e) part[t * kRP + r] = fmaf(qf[r][m * C::kEPC + e], f[e], part[t * kRP + r]);
        }
      }
      const float s = group_transpose_sum(part, lane);
      const int key = wkb + rnd * kKeysPerRound + grp * kTPR + (j / kRP);
      sc[rnd] = key < vis_row ? s : -CUDART_INF_F;
    }

    // ---- online softmax for row `myrow` (lanes with equal lane % 4)
    float mx = sc[0];
#pragma unroll
    for (int rnd = 1; rnd < kRounds; ++rnd) mx = fmaxf(mx, sc[rnd]);
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
    const float m_new = fmaxf(m_row, mx);
    const float m_use = m_new == -CUDART_INF_F ? 0.f : m_new;
    const float alpha = exp2f(m_row - m_use);
    float psum = 0.f;
#pragma unroll
    for (int rnd = 0; rnd < kRounds; ++rnd) {
      const float pr = exp2f(sc[rnd] - m_use);
      psum += pr;
      pw[(rnd * kKeysPerRound + grp * kTPR + (j / kRP)) * kRP + myrow] = pr;
    }
    psum += __shfl_xor_sync(0xffffffffu, psum, 4);
    psum += __shfl_xor_sync(0xffffffffu, psum, 8);
    psum += __shfl_xor_sync(0xffffffffu, psum, 16);
    l_row = l_row * alpha + psum;
    m_row = m_new;
    float a[kRP];
#pragma unroll
    for (int r = 0; r < kRP; ++r) a[r] = __shfl_sync(0xffffffffu, alpha, r);
#pragma unroll
    for (int r = 0; r < kRP; ++r)
#pragma unroll
      for (int e = 0; e < C::kDPL; ++e) acc[r][e] *= a[r];
    __syncwarp();

    // ---- acc += P V over this warp's keys that exist (keys >= ke may hold garbage)
    const int kcount = max(0, min(kWarpKeys, it.ke - wkb));
#pragma unroll
    for (int kk = 0; kk < kWarpKeys; ++kk) {
      if (kk < kcount) {
        const float4 pv = *reinterpret_cast<const float4*>(pw + kk * kRP);
        float vf[C::kDPL];
        load_v<T, C::kDPL>(vs + kk * C::kRowBytes + lane * C::kDPL * C::kEs, vf);
#pragma unroll
        for (int e = 0; e < C::kDPL; ++e) {
          acc[0][e] = fmaf(pv.x, vf[e], acc[0][e]);
          acc[1][e] = fmaf(pv.y, vf[e], acc[1][e]);
          acc[2][e] = fmaf(pv.z, vf[e], acc[2][e]);
          acc[3][e] = fmaf(pv.w, vf[e], acc[3][e]);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[stage]);
    ++tile;

    if (mt.flags & kMetaLast) {
      // ---- merge the 4 warp states and write the item's rows
      if (lane < kRP) {
        comb_ml[(warp * kRP + lane) * 2 + 0] = m_row;
        comb_ml[(warp * kRP + lane) * 2 + 1] = l_row;
      }
#pragma unroll
      for (int r = 0; r < kRP; ++r)
#pragma unroll
        for (int e = 0; e < C::kDPL; ++e) comb_acc[(warp * kRP + r) * D + lane * C::kDPL + e] = acc[r][e];
      named_barrier(1, kConsumerWarps * 32);
      for (int idx = threadIdx.x; idx < kRP * D; idx += kConsumerWarps * 32) {
        const int r = idx / D, d = idx - r * D;
        if (r >= it.nrows) continue;
        float M = -CUDART_INF_F;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, comb_ml[(w * kRP + r) * 2]);
        const float Mu = M == -CUDART_INF_F ? 0.f : M;
        float lsum = 0.f, o = 0.f;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) {
          const float wt = exp2f(comb_ml[(w * kRP + r) * 2] - Mu);
          lsum = fmaf(wt, comb_ml[(w * kRP + r) * 2 + 1], lsum);
          o = fmaf(wt, comb_acc[(w * kRP + r) * D + d], o);
        }
        if (it.part < 0) {
          const int row = it.row0 + r;
          const int tok = row / p.G, g = row - tok * p.G;
          T* orow = reinterpret_cast<T*>(p.out) + ((int64_t)(qstart + tok) * p.Hq + (int64_t)it.kvh * p.G + g) * D;
          orow[d] = Elem<T>::to_out(o / lsum);
        } else {
          p.part_acc[(int64_t)(it.part + r) * D + d] = o;
          if (d == 0) p.part_ml[it.part + r] = make_float2(M, lsum);
        }
      }
      named_barrier(1, kConsumerWarps * 32);
    }
  }
}

template <typename T, int D>
__global__ void __launch_bounds__(128) merge_kernel(const MergeParams p) {
  const int n = p.header->n_merge;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int gi = blockIdx.x; gi < n; gi += gridDim.x) {
    const MergeGroup g = p.groups[gi];
    const int qstart = p.query_start_loc[g.seq];
    for (int r = warp; r < g.nrows; r += 4) {
      float M = -CUDART_INF_F;
      for (int sp = 0; sp < g.nsplit; ++sp) M = fmaxf(M, p.part_ml[g.part_base + sp * g.nrows + r].x);
      const float Mu = M == -CUDART_INF_F ? 0.f : M;
      float lsum = 0.f;
      for (int sp = 0; sp < g.nsplit; ++sp) {
        const float2 ml = p.part_ml[g.part_base + sp * g.nrows + r];
        lsum = fmaf(exp2f(ml.x - Mu), ml.y, lsum);
      }
      const float inv = 1.f / lsum;
      const int row = g.row0 + r;
      const int tok = row / p.G, gg = row - tok * p.G;
      T* orow = reinterpret_cast<T*>(p.out) + ((int64_t)(qstart + tok) * p.Hq + (int64_t)g.kvh * p.G + gg) * D;
      for (int d = lane; d < D; d += 32) {
        float o = 0.f;
        for (int sp = 0; sp < g.nsplit; ++sp) {
          const int slot = g.part_base + sp * g.nrows + r;
          o = fmaf(exp2f(p.part_ml[slot].x - Mu), p.part_acc[(int64_t)slot * D + d], o);
        }
        orow[d] = Elem<T>::to_out(o * inv);
      }
    }
  }
}

// The dynamic shared-memory opt-in is a per-device function attribute.
template <typename T, int D>
cudaError_t prepare_decode(int* ctas_per_sm) {
  using C = Cfg<T, D>;
  static unsigned long long done_mask = 0;  // one bit per device ordinal (< 64)
  static int occupancy[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!(__atomic_load_n(&done_mask, __ATOMIC_ACQUIRE) & (1ull << dev))) {
    e = cudaFuncSetAttribute(decode_kernel<T, D>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
    if (e != cudaSuccess) return e;
    int occ = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, decode_kernel<T, D>, kThreads, C::kSmem);
    if (e != cudaSuccess) return e;
    occupancy[dev] = occ < 1 ? 1 : occ;
    __atomic_fetch_or(&done_mask, 1ull << dev, __ATOMIC_RELEASE);
  }
  if (ctas_per_sm) *ctas_per_sm = occupancy[dev];
  return cudaSuccess;
}

template <typename T, int D>
cudaError_t launch_decode_t(const AttnParams& p, const CUtensorMap& kmap, const CUtensorMap& vmap, int grid,
                            cudaStream_t s) {
  using C = Cfg<T, D>;
  cudaError_t e = prepare_decode<T, D>(nullptr);
  if (e != cudaSuccess) return e;
  decode_kernel<T, D><<<grid, kThreads, C::kSmem, s>>>(p, kmap, vmap);
  return cudaGetLastError();
}

}  // namespace

cudaError_t decode_ctas_per_sm(bool bf16, int D, int* ctas) {
  if (bf16) return D == 128 ? prepare_decode<__nv_bfloat16, 128>(ctas) : prepare_decode<__nv_bfloat16, 64>(ctas);
  return D == 128 ? prepare_decode<float, 128>(ctas) : prepare_decode<float, 64>(ctas);
}

int decode_smem_bytes(int D, int elem_bytes) {
  if (elem_bytes == 2) return D == 128 ? Cfg<__nv_bfloat16, 128>::kSmem : Cfg<__nv_bfloat16, 64>::kSmem;
  return D == 128 ? Cfg<float, 128>::kSmem : Cfg<float, 64>::kSmem;
}

cudaError_t launch_decode(const AttnParams& p, const CUtensorMap& kmap, const CUtensorMap& vmap, bool bf16, int grid,
                          cudaStream_t s) {
  if (bf16) {
    return p.D == 128 ? launch_decode_t<__nv_bfloat16, 128>(p, kmap, vmap, grid, s)
                      : launch_decode_t<__nv_bfloat16, 64>(p, kmap, vmap, grid, s);
  }
  return p.D == 128 ? launch_decode_t<float, 128>(p, kmap, vmap, grid, s)
                    : launch_decode_t<float, 64>(p, kmap, vmap, grid, s);
}

cudaError_t launch_merge(const MergeParams& p, bool bf16, int grid, cudaStream_t s) {
  if (bf16) {
    if (p.D == 128)
      merge_kernel<__nv_bfloat16, 128><<<grid, 128, 0, s>>>(p);
    else
      merge_kernel<__nv_bfloat16, 64><<<grid, 128, 0, s>>>(p);
  } else {
    if (p.D == 128)
      merge_kernel<float, 128><<<grid, 128, 0, s>>>(p);
    else
      merge_kernel<float, 64><<<grid, 128, 0, s>>>(p);
  }
  return cudaGetLastError();
}

}  // namespace pkv
