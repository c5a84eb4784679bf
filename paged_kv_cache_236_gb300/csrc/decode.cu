// CUDA-core paged attention for few rows per kv head (decode), with split-KV.
//
// What it computes ("Paged Attention 基础", section 2, steps 1-5): for each
// work item - up to kDecRows rows (query token, head-in-group) of one
// sequence and one kv head, over keys [kb, ke) - walk the block table, fetch
// each key block, form scale * q.k, apply the causal mask at the query's
// absolute position L - n + i, and accumulate softmax(.)V with a running
// (max, sum) ("online softmax").  Items that cover a whole key range write
// normalised output rows.  Split items write partial (m, l, acc) rows; the
// last split of a merge group to finish (an atomic ticket, no waiting)
// combines them: m = max_p m_p, l = sum_p l_p 2^(m_p - m),
// O = sum_p acc_p 2^(m_p - m) / l (logits kept in log2 units).
//
// GB300 design:
//  * persistent CTAs (2 per SM) take items from an atomic counter, in the
//    planner's largest-first order;
//  * a producer warp streams each 64-key tile of K and V with TMA: one 4-D
//    tensor-map box per physical block ({head_dim, 1 head, block_size, 1
//    block} of the pool [num_blocks, block_size, num_kv_heads, head_dim]), so
//    the block table is resolved by the box coordinate and blocks past a
//    sequence's end (or invalid ids) are out-of-range boxes that read as
//    zeros.  Block ids are loaded one tile ahead; an item's q rows arrive in
//    the same stage as its first tile (bulk copies); the item's description
//    travels in the stage's metadata, so consumers never wait on global
//    memory.  A 3-stage mbarrier ring keeps ~64 KB per CTA in flight;
//  * 4 consumer warps each own 16 keys of a tile: 8 lanes per key (16-byte
//    shared loads, conflict-free), partial dot products for the 4 rows of 2
//    keys in packed fp32x2 FMAs reduced with a transposing butterfly (7
//    shuffles per 8 scores), warp-level online softmax, then P.V with each
//    lane owning head_dim/32 output columns of all 4 rows (packed FMAs); the
//    4 warp states are merged at the end of an item through shared memory.
#include <cuda_fp8.h>
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
constexpr int kMetaDone = 2, kMetaLast = 1, kMetaFirst = 4;
static_assert(kRP == 4 && kLPT == 8, "butterfly below is written for 8 partials per lane");

// T: the element of q and out; KV: the element of the K and V pools (T, or
// E4M3 codes for the FP8 cache, read as fp32 code values; the scales are
// folded into the logit scale and applied to the output).
template <typename T, typename KV, int D>
struct Cfg {
  static constexpr int kEs = sizeof(T);
  static constexpr int kKvEs = sizeof(KV);
  static constexpr int kQRowBytes = D * kEs;
  static constexpr int kRowBytes = D * kKvEs;  // one K or V row
  static constexpr int kChunks = kRowBytes / 16;
  static constexpr int kCPL = kChunks / kLPT;  // 16-byte K chunks per lane per key
  static constexpr int kEPC = 16 / kKvEs;      // K elements per chunk
  static constexpr int kEPL = kCPL * kEPC;     // q elements per lane
  static constexpr int kQCPC = kEPC * kEs / 16;  // 16-byte q chunks per K chunk
  static constexpr int kDPL = D / 32;          // output columns per lane
  static constexpr int kTileBytes = kDecTileKeys * kRowBytes;
  static constexpr int kQSlotOff = 2 * kTileBytes;  // an item's q rows, in its first tile's stage
  static constexpr int kStageBytes = (2 * kTileBytes + kRP * kQRowBytes + 1023) / 1024 * 1024;
  static constexpr int kStages =
      (98304 / kStageBytes) < 2 ? 2 : ((98304 / kStageBytes) > 4 ? 4 : (98304 / kStageBytes));
  // shared memory carve-up
  static constexpr int kPOff = kStages * kStageBytes;
  static constexpr int kPBytes = kConsumerWarps * kWarpKeys * kRP * 8;  // (p, p) pairs
  static constexpr int kAccOff = kPOff + kPBytes;
  static constexpr int kAccBytes = kConsumerWarps * kRP * D * 4;
  static constexpr int kMlOff = kAccOff + kAccBytes;
  static constexpr int kMlBytes = kConsumerWarps * kRP * 2 * 4;
  static constexpr int kMetaOff = kMlOff + kMlBytes;
  static constexpr int kMetaBytes = kStages * 64;
  static constexpr int kBarOff = kMetaOff + kMetaBytes;
  static constexpr int kSmem = kBarOff + 2 * kStages * 8 + 16 + 1024;  // + slack to align the base to 1 KB
  static_assert(kCPL >= 1 && kChunks % kLPT == 0, "row must split into 8 lanes of 16-byte chunks");
  static_assert(kQCPC >= 1, "q elements of a K chunk fill whole 16-byte chunks");
};

// What a stage carries besides K and V: which item and key tile, and the
// item's description (so consumers need no global loads).
struct alignas(16) Meta {
  int item, kbase, flags, seq;
  int kvh, row0, nrows, ke;
  int part, grp, L, n;
  int qstart, pad0, pad1, pad2;
};
static_assert(sizeof(Meta) == 64, "meta slot");

// One 16-byte chunk of K or q as kEPC/2 fp32 pairs (elements 2j, 2j+1).
template <typename T>
__device__ __forceinline__ void chunk_to_pairs(const uint4 raw, f32x2* f);
template <>
__device__ __forceinline__ void chunk_to_pairs<__nv_bfloat16>(const uint4 raw, f32x2* f) {
  f[0] = pk2(bf16_lo(raw.x), bf16_hi(raw.x));
  f[1] = pk2(bf16_lo(raw.y), bf16_hi(raw.y));
  f[2] = pk2(bf16_lo(raw.z), bf16_hi(raw.z));
  f[3] = pk2(bf16_lo(raw.w), bf16_hi(raw.w));
}
template <>
__device__ __forceinline__ void chunk_to_pairs<float>(const uint4 raw, f32x2* f) {
  f[0] = pk2(__uint_as_float(raw.x), __uint_as_float(raw.y));
  f[1] = pk2(__uint_as_float(raw.z), __uint_as_float(raw.w));
}
// Two E4M3 codes (low byte first) as their fp32 values (exact: E4M3 values
// are fp16 values).
__device__ __forceinline__ f32x2 e4m3x2_to_pair(uint32_t two) {
  const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)two, __NV_E4M3);
  const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h));
  return pk2(f.x, f.y);
}
template <>
__device__ __forceinline__ void chunk_to_pairs<__nv_fp8_e4m3>(const uint4 raw, f32x2* f) {
  const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = e4m3x2_to_pair(w[i] & 0xFFFFu);
    f[2 * i + 1] = e4m3x2_to_pair(w[i] >> 16);
  }
}

// This lane's kDPL V columns of one key row as fp32 pairs.
template <typename T, int DPL>
__device__ __forceinline__ void load_v_pairs(const uint8_t* p, f32x2* f) {
  if constexpr (sizeof(T) == 1) {
    if constexpr (DPL == 4) {
      const uint32_t w = *reinterpret_cast<const uint32_t*>(p);
      f[0] = e4m3x2_to_pair(w & 0xFFFFu);
      f[1] = e4m3x2_to_pair(w >> 16);
    } else {
      f[0] = e4m3x2_to_pair(*reinterpret_cast<const uint16_t*>(p));
    }
  } else if constexpr (sizeof(T) == 2) {
    if constexpr (DPL == 4) {
      const uint2 w = *reinterpret_cast<const uint2*>(p);
      f[0] = pk2(bf16_lo(w.x), bf16_hi(w.x));
      f[1] = pk2(bf16_lo(w.y), bf16_hi(w.y));
    } else {
      const uint32_t w = *reinterpret_cast<const uint32_t*>(p);
      f[0] = pk2(bf16_lo(w), bf16_hi(w));
    }
  } else {
    if constexpr (DPL == 4) {
      const uint4 w = *reinterpret_cast<const uint4*>(p);
      f[0] = pk2(__uint_as_float(w.x), __uint_as_float(w.y));
      f[1] = pk2(__uint_as_float(w.z), __uint_as_float(w.w));
    } else {
      const uint2 w = *reinterpret_cast<const uint2*>(p);
      f[0] = pk2(__uint_as_float(w.x), __uint_as_float(w.y));
    }
  }
}

// Sum v[i] over the 8 lanes of a lane group, transposing: afterwards lane
// (lane & 7) == i holds the group total of v[i].
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

__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_u32(dst)),
               "l"(src), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}

template <typename T, typename KV, int D>
__global__ void __launch_bounds__(kThreads, 2) decode_kernel(const AttnParams p,
                                                             const __grid_constant__ CUtensorMap kmap,
                                                             const __grid_constant__ CUtensorMap vmap) {
  using C = Cfg<T, KV, D>;
  extern __shared__ __align__(16) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  f32x2* pbuf = reinterpret_cast<f32x2*>(smem + C::kPOff);
  float* comb_acc = reinterpret_cast<float*>(smem + C::kAccOff);
  float* comb_ml = reinterpret_cast<float*>(smem + C::kMlOff);
  Meta* meta = reinterpret_cast<Meta*>(smem + C::kMetaOff);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::kBarOff);
  uint64_t* empty = full + C::kStages;
  int* flag_last = reinterpret_cast<int*>(empty + C::kStages);
  const WaitCtl wc{p.err, wait_limit(p.wait_ns)};

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kConsumerWarps);
    }
    fence_mbar_init();
  }
  __syncthreads();
  pdl_wait();  // the plan and the K/V write are complete and visible from here on
  const int n_items = p.header->n_dec;

  if (warp == kConsumerWarps) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tensormap(&kmap);
      prefetch_tensormap(&vmap);
    }
    const int nb_per_tile = kDecTileKeys / p.bs;
    int tile = 0;
    // On giving up: wait (bounded) until the copies of the last tiles
    // issued have landed, so that none is still in
    // flight into this CTA's shared memory when it exits.
    auto drain = [&]() {
      for (int j = max(0, tile - C::kStages); j < tile; ++j)
        __all_sync(0xffffffffu, mbar_wait(&full[j % C::kStages], (j / C::kStages) & 1, wc));
    };
    int idx = 0;
    if (lane == 0) idx = atomicAdd(p.counter, 1);
    idx = __shfl_sync(0xffffffffu, idx, 0);
    for (;;) {
      if (idx >= n_items) {
        const int stage = tile % C::kStages;
        if (!__all_sync(0xffffffffu, mbar_wait(&empty[stage], ((tile / C::kStages) & 1) ^ 1, wc))) {
          drain();
          return;
        }
        if (lane == 0) {
          meta[stage].item = -1;
          meta[stage].flags = kMetaDone;
          mbar_arrive(&full[stage]);
        }
        break;
      }
      const WorkItem it = p.items[idx];
      // take the next item now; its index is only needed after this item's tiles
      int next = 0;
      if (lane == 0) next = atomicAdd(p.counter, 1);
      const int L = p.context_lens[it.seq];
      const int qstart = p.query_start_loc[it.seq];
      const int n = p.query_start_loc[it.seq + 1] - qstart;
      const int nblk = (L + p.bs - 1) / p.bs;
      const int32_t* bt = p.block_tables + (int64_t)it.seq * p.max_blocks;
      auto block_of = [&](int kbase) -> int {  // physical block for this lane in the tile at kbase
        const int lb = kbase / p.bs + lane;
        int phys = (int)p.num_blocks;  // out of range: the box reads as zeros
        if (lane < nb_per_tile && lb < nblk) {
          const int b = __ldg(bt + lb);
          if (b >= 0 && (int64_t)b < p.num_blocks)
            phys = b;
          else
            raise_error(p.err, PKV_DEVERR_BLOCK_OUT_OF_RANGE);
        }
        return phys;
      };
      int phys = block_of(it.kb);
      for (int kbase = it.kb; kbase < it.ke; kbase += kDecTileKeys) {
        const int stage = tile % C::kStages;
        const bool first = kbase == it.kb;
        const int next_phys = (kbase + kDecTileKeys < it.ke) ? block_of(kbase + kDecTileKeys) : 0;
        if (!__all_sync(0xffffffffu, mbar_wait(&empty[stage], ((tile / C::kStages) & 1) ^ 1, wc))) {
          drain();
          return;
        }
        if (p.fault_tile == tile + 1 && blockIdx.x == 0) {
          // testing only: this tile is never loaded, so its consumers' waits run out
          phys = next_phys;
          ++tile;
          continue;
        }
        uint8_t* sbase = smem + stage * C::kStageBytes;
        if (lane == 0) {
          Meta& m = meta[stage];
          m.item = idx;
          m.kbase = kbase;
          m.flags = ((kbase + kDecTileKeys >= it.ke) ? kMetaLast : 0) | (first ? kMetaFirst : 0);
          m.seq = it.seq;
          m.kvh = it.kvh;
          m.row0 = it.row0;
          m.nrows = it.nrows;
          m.ke = it.ke;
          m.part = it.part;
          m.grp = it.grp;
          m.L = L;
          m.n = n;
          m.qstart = qstart;
          mbar_arrive_expect_tx(&full[stage], 2 * C::kTileBytes + (first ? it.nrows * C::kQRowBytes : 0));
        }
        __syncwarp();
        if (lane < nb_per_tile) {
          uint8_t* kdst = sbase + lane * p.bs * C::kRowBytes;
          tma_load_4d(kdst, &kmap, &full[stage], 0, it.kvh, 0, phys);
          tma_load_4d(kdst + C::kTileBytes, &vmap, &full[stage], 0, it.kvh, 0, phys);
        }
        if (first && lane < it.nrows) {
          const int row = it.row0 + lane;
          const int tok = row / p.G, g = row - tok * p.G;
          const T* qrow =
              reinterpret_cast<const T*>(p.q) + ((int64_t)(qstart + tok) * p.Hq + (int64_t)it.kvh * p.G + g) * D;
          bulk_load(sbase + C::kQSlotOff + lane * C::kQRowBytes, qrow, C::kQRowBytes, &full[stage]);
        }
        phys = next_phys;
        ++tile;
      }
      idx = __shfl_sync(0xffffffffu, next, 0);
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const int grp = lane >> 3, j = lane & 7;
  const int myrow = lane & (kRP - 1);  // row whose scores this lane holds
  f32x2* pw = pbuf + warp * kWarpKeys * kRP;

  f32x2 qf[kRP][C::kEPL / 2];
  f32x2 acc[kRP][C::kDPL / 2];
  float m_row = -CUDART_INF_F, l_row = 0.f;
  int vis_row = 0;  // keys visible to row `myrow` (absolute key < vis_row)
  int tile = 0;
  for (;;) {
    const int stage = tile % C::kStages;
    // The four consumer warps wait for the same tile; they agree before going
    // on, so that if one gave up, all leave (none is left waiting alone at
    // the item's end barrier).
    const bool got = __all_sync(0xffffffffu, mbar_wait(&full[stage], (tile / C::kStages) & 1, wc));
    if (barrier_any(3, kConsumerWarps * 32, !got)) break;
    const Meta mt = meta[stage];
    if (mt.flags & kMetaDone) break;
    const uint8_t* sbase = smem + stage * C::kStageBytes;
    if (mt.flags & kMetaFirst) {
      m_row = -CUDART_INF_F;
      l_row = 0.f;
      const f32x2 sc2 = pk2(p.scale_log2, p.scale_log2);
#pragma unroll
      for (int r = 0; r < kRP; ++r) {
#pragma unroll
        for (int e = 0; e < C::kDPL / 2; ++e) acc[r][e] = 0ull;
        if (r < mt.nrows) {
          const uint8_t* qrow = sbase + C::kQSlotOff + r * C::kQRowBytes;
          // this lane's q elements: the kEPC elements of each of its K chunks
#pragma unroll
          for (int m = 0; m < C::kCPL; ++m) {
#pragma unroll
            for (int u = 0; u < C::kQCPC; ++u) {
              const uint4 raw = *reinterpret_cast<const uint4*>(qrow + ((j + 8 * m) * C::kQCPC + u) * 16);
              constexpr int kQP = 8 / C::kEs;  // fp32 pairs in a 16-byte q chunk
              f32x2 f[kQP];
              chunk_to_pairs<T>(raw, f);
#pragma unroll
              for (int e = 0; e < kQP; ++e) qf[r][m * (C::kEPC / 2) + u * kQP + e] = mul2(f[e], sc2);
            }
          }
        } else {
#pragma unroll
          for (int e = 0; e < C::kEPL / 2; ++e) qf[r][e] = 0ull;
        }
      }
      const int tok = (mt.row0 + myrow) / p.G;
      vis_row = myrow < mt.nrows ? min(mt.ke, p.causal ? mt.L - mt.n + tok + 1 : mt.L) : 0;
    }
    const uint8_t* ks = sbase + warp * kWarpKeys * C::kRowBytes;
    const uint8_t* vs = ks + C::kTileBytes;
    const int wkb = mt.kbase + warp * kWarpKeys;  // absolute key of this warp's first key

    // ---- scores: s = (scale*log2e) q.k for 4 rows x 16 keys, 2 per lane
    float sc[kRounds];
#pragma unroll
    for (int rnd = 0; rnd < kRounds; ++rnd) {
      f32x2 part2[kTPR * kRP];
#pragma unroll
      for (int i = 0; i < kTPR * kRP; ++i) part2[i] = 0ull;
#pragma unroll
      for (int t = 0; t < kTPR; ++t) {
        const int kl = rnd * kKeysPerRound + grp * kTPR + t;
        const uint8_t* krow = ks + kl * C::kRowBytes;
#pragma unroll
        for (int m = 0; m < C::kCPL; ++m) {
          const uint4 raw = *reinterpret_cast<const uint4*>(krow + (j + 8 * m) * 16);
          f32x2 f[C::kEPC / 2];
          chunk_to_pairs<KV>(raw, f);
#pragma unroll
          for (int r = 0; r < kRP; ++r)
#pragma unroll
            for (int e = 0; e < C::kEPC / 2; ++e)
              part2[t * kRP + r] = fma2(qf[r][m * (C::kEPC / 2) + e], f[e], part2[t * kRP + r]);
        }
      }
      float part[kTPR * kRP];
#pragma unroll
      for (int i = 0; i < kTPR * kRP; ++i) {
        const float2 h = up2(part2[i]);
        part[i] = h.x + h.y;
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
      pw[(rnd * kKeysPerRound + grp * kTPR + (j / kRP)) * kRP + myrow] = pk2(pr, pr);
    }
    psum += __shfl_xor_sync(0xffffffffu, psum, 4);
    psum += __shfl_xor_sync(0xffffffffu, psum, 8);
    psum += __shfl_xor_sync(0xffffffffu, psum, 16);
    l_row = l_row * alpha + psum;
    m_row = m_new;
#pragma unroll
    for (int r = 0; r < kRP; ++r) {
      const float a = __shfl_sync(0xffffffffu, alpha, r);
      const f32x2 a2 = pk2(a, a);
#pragma unroll
      for (int e = 0; e < C::kDPL / 2; ++e) acc[r][e] = mul2(acc[r][e], a2);
    }
    __syncwarp();

    // ---- acc += P V over this warp's keys that exist (keys >= ke may hold garbage)
    const int kcount = max(0, min(kWarpKeys, mt.ke - wkb));
#pragma unroll
    for (int kk = 0; kk < kWarpKeys; ++kk) {
      if (kk < kcount) {
        const ulonglong2 p01 = *reinterpret_cast<const ulonglong2*>(pw + kk * kRP);
        const ulonglong2 p23 = *reinterpret_cast<const ulonglong2*>(pw + kk * kRP + 2);
        const f32x2 pp[4] = {p01.x, p01.y, p23.x, p23.y};
        f32x2 vf[C::kDPL / 2];
        load_v_pairs<KV, C::kDPL>(vs + kk * C::kRowBytes + lane * C::kDPL * C::kKvEs, vf);
#pragma unroll
        for (int r = 0; r < kRP; ++r)
#pragma unroll
          for (int e = 0; e < C::kDPL / 2; ++e) acc[r][e] = fma2(pp[r], vf[e], acc[r][e]);
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
        for (int e = 0; e < C::kDPL / 2; ++e) {
          const float2 h = up2(acc[r][e]);
          comb_acc[(warp * kRP + r) * D + lane * C::kDPL + 2 * e] = h.x;
          comb_acc[(warp * kRP + r) * D + lane * C::kDPL + 2 * e + 1] = h.y;
        }
      named_barrier(1, kConsumerWarps * 32);
      for (int idx = threadIdx.x; idx < kRP * D; idx += kConsumerWarps * 32) {
        const int r = idx / D, d = idx - r * D;
        if (r >= mt.nrows) continue;
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
        if (mt.part < 0) {
          const int row = mt.row0 + r;
          const int tok = row / p.G, g = row - tok * p.G;
          T* orow =
              reinterpret_cast<T*>(p.out) + ((int64_t)(mt.qstart + tok) * p.Hq + (int64_t)mt.kvh * p.G + g) * D;
          orow[d] = Elem<T>::to_out(o / lsum * p.v_scale);
        } else {
          p.part_acc[(int64_t)(mt.part + r) * D + d] = o;
          if (d == 0) p.part_ml[mt.part + r] = make_float2(M, lsum);
        }
      }
      if (mt.part >= 0) {
        // the split that completes its merge group combines the group's partials
        __threadfence();
        named_barrier(1, kConsumerWarps * 32);
        if (threadIdx.x == 0) *flag_last = atomicAdd(p.tickets + mt.grp, 1);
        named_barrier(1, kConsumerWarps * 32);
        const MergeGroup g = p.groups[mt.grp];
        if (*flag_last == g.nsplit - 1) {
          __threadfence();
          for (int idx = threadIdx.x; idx < g.nrows * D; idx += kConsumerWarps * 32) {
            const int r = idx / D, d = idx - r * D;
            float M = -CUDART_INF_F;
#pragma unroll 8
            for (int sp = 0; sp < g.nsplit; ++sp)
              M = fmaxf(M, __ldcg(&p.part_ml[g.part_base + sp * g.nrows + r]).x);
            const float Mu = M == -CUDART_INF_F ? 0.f : M;
            float lsum = 0.f, o = 0.f;
#pragma unroll 8
            for (int sp = 0; sp < g.nsplit; ++sp) {
              const int slot = g.part_base + sp * g.nrows + r;
              const float2 ml = __ldcg(&p.part_ml[slot]);
              const float wt = exp2f(ml.x - Mu);
              lsum = fmaf(wt, ml.y, lsum);
              o = fmaf(wt, __ldcg(&p.part_acc[(int64_t)slot * D + d]), o);
            }
            const int row = g.row0 + r;
            const int tok = row / p.G, gh = row - tok * p.G;
            T* orow =
                reinterpret_cast<T*>(p.out) + ((int64_t)(mt.qstart + tok) * p.Hq + (int64_t)g.kvh * p.G + gh) * D;
            orow[d] = Elem<T>::to_out(o / lsum * p.v_scale);
          }
        }
      }
      named_barrier(1, kConsumerWarps * 32);
    }
  }
}

// The dynamic shared-memory opt-in is a per-device function attribute.
template <typename T, typename KV, int D>
cudaError_t prepare_decode(int* ctas_per_sm) {
  using C = Cfg<T, KV, D>;
  static unsigned long long done_mask = 0;  // one bit per device ordinal (< 64)
  static int occupancy[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!(__atomic_load_n(&done_mask, __ATOMIC_ACQUIRE) & (1ull << dev))) {
    e = cudaFuncSetAttribute(decode_kernel<T, KV, D>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
    if (e != cudaSuccess) return e;
    int occ = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, decode_kernel<T, KV, D>, kThreads, C::kSmem);
    if (e != cudaSuccess) return e;
    occupancy[dev] = occ < 1 ? 1 : occ;
    __atomic_fetch_or(&done_mask, 1ull << dev, __ATOMIC_RELEASE);
  }
  if (ctas_per_sm) *ctas_per_sm = occupancy[dev];
  return cudaSuccess;
}

template <typename T, typename KV, int D>
cudaError_t launch_decode_t(const AttnParams& p, const CUtensorMap& kmap, const CUtensorMap& vmap, int grid,
                            cudaStream_t s) {
  using C = Cfg<T, KV, D>;
  cudaError_t e = prepare_decode<T, KV, D>(nullptr);
  if (e != cudaSuccess) return e;
  e = launch_pdl(decode_kernel<T, KV, D>, dim3(grid), dim3(kThreads), C::kSmem, s, p, kmap, vmap);
  return e != cudaSuccess ? e : cudaGetLastError();
}

using bf16_t = __nv_bfloat16;
using e4m3_t = __nv_fp8_e4m3;

}  // namespace

cudaError_t decode_ctas_per_sm(bool bf16, int D, int* ctas) {
  if (bf16) return D == 128 ? prepare_decode<bf16_t, bf16_t, 128>(ctas) : prepare_decode<bf16_t, bf16_t, 64>(ctas);
  return D == 128 ? prepare_decode<float, float, 128>(ctas) : prepare_decode<float, float, 64>(ctas);
}

cudaError_t decode_fp8_ctas_per_sm(int* ctas) { return prepare_decode<bf16_t, e4m3_t, 128>(ctas); }

int decode_smem_bytes(int D, int elem_bytes) {
  if (elem_bytes == 2) return D == 128 ? Cfg<bf16_t, bf16_t, 128>::kSmem : Cfg<bf16_t, bf16_t, 64>::kSmem;
  return D == 128 ? Cfg<float, float, 128>::kSmem : Cfg<float, float, 64>::kSmem;
}

cudaError_t launch_decode(const AttnParams& p, const CUtensorMap& kmap, const CUtensorMap& vmap, bool bf16, int grid,
                          cudaStream_t s) {
  if (bf16) {
    return p.D == 128 ? launch_decode_t<bf16_t, bf16_t, 128>(p, kmap, vmap, grid, s)
                      : launch_decode_t<bf16_t, bf16_t, 64>(p, kmap, vmap, grid, s);
  }
  return p.D == 128 ? launch_decode_t<float, float, 128>(p, kmap, vmap, grid, s)
                    : launch_decode_t<float, float, 64>(p, kmap, vmap, grid, s);
}

cudaError_t launch_decode_fp8(const AttnParams& p, const CUtensorMap& kmap, const CUtensorMap& vmap, int grid,
                              cudaStream_t s) {
  return launch_decode_t<bf16_t, e4m3_t, 128>(p, kmap, vmap, grid, s);
}

}  // namespace pkv
