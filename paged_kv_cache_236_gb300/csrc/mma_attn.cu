// Tensor-core paged attention for multi-token queries (prefill chunks,
// speculative verification): tcgen05.mma with TMEM accumulators.
//
// What it computes is the same as the other attention kernels ("Paged
// Attention 基础", section 2, steps 1-5; causal mask at each query's absolute
// position L - n + i; "ADR 004" Consequences: prefill and decode share one
// call), for a work item of up to 128 rows (query token, head-in-group) of one
// sequence and one kv head over keys [kb, ke):
//   S = Q K^T (128 rows x 64 keys per tile, fp32 in TMEM), online softmax in
//   registers, P (bf16) -> shared memory, O += P V (fp32 in TMEM), O / l at
//   the end, or a partial (m, l, O) row for split-KV; the last split of a
//   merge group to finish merges the group (atomic ticket, no waiting).
//
// Roles (320 threads, one CTA per SM, persistent over items):
//   warp 0    TMA producer: the item's Q tile (3-D box {64, G heads, 128/G
//             tokens} of q [T, Hq, D], two 64-column halves) and, per 64-key
//             tile, one {64, 1, block_size, 1} box per physical block and
//             64-column half of the pool [NB, bs, Hkv, D] for K and for V
//             (128-byte swizzle, the layout the tensor core reads); block ids
//             are loaded one tile ahead;
//   warp 1    TMEM allocation and the single thread issuing the MMAs; the
//             P.V of tile g is issued after the S of tile g+1;
//   warps 2-9 softmax / correction / epilogue: two threads per row (TMEM
//             lane), warps 2-5 on key columns 0-31 of a tile, warps 6-9 on
//             32-63; a pair exchanges row maxima (and at the end row sums)
//             through shared memory.
// Shared memory: Q 32 KB, a 5-stage ring of K+V tiles (160 KB), 2 P buffers
// (32 KB).  TMEM: S double-buffered in columns [0,128), O in [128,256).
//
// The running max used for the exponentials is only raised when a tile's row
// maximum exceeds it by more than 8 (log2 units), so O is rescaled in TMEM
// rarely; P stays <= 2^8 and the result is exact up to rounding.
#include <math_constants.h>

#include "pkv_device.cuh"
#include "pkv_internal.h"
#include "pkv_tc.cuh"

namespace pkv {
namespace {

constexpr int kThreads = 320;
constexpr int kKeys = 64;                           // keys per tile
constexpr int kStages = 5;
constexpr int kHalfKV = kKeys * 128;                // one 64-column half of a K or V tile (8 KB)
constexpr int kTileBytes = 2 * kHalfKV;             // K or V tile: 16 KB
constexpr int kStageBytes = 2 * kTileBytes;         // K + V: 32 KB
constexpr int kQBytes = kMmaRows * 128 * 2;         // 32 KB (two 16 KB halves)
constexpr int kPBytes = kMmaRows * kKeys * 2;       // 16 KB
// shared-memory carve-up (offsets from a 1024-byte aligned base)
constexpr int kQOff = 0;
constexpr int kSOff = kQOff + kQBytes;              // stages: K tile then V tile
constexpr int kPOff = kSOff + kStages * kStageBytes;
constexpr int kBarOff = kPOff + 2 * kPBytes;
constexpr int kNumBars = 2 + 3 * kStages + 2 * 4 + 2;
constexpr int kRedOff = kBarOff + kNumBars * 8 + 16;  // [2 tiles][2 halves][128 rows] row maxima / sums
// No alignment slack: the buffers need a 1024-byte aligned base, which the
// dynamic shared memory of a kernel without static shared memory has; the
// kernel checks and refuses to run otherwise.
constexpr int kSmem = kRedOff + 2 * 2 * 128 * 4;
constexpr uint32_t kTmemCols = 256;
constexpr uint32_t kSCol = 0, kOCol = 128;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

constexpr uint32_t kIdescS = idesc_bf16(128, kKeys, false, false);
constexpr uint32_t kIdescO = idesc_bf16(128, 128, false, true);

// V as the B of P.V (MN-major): the two 64-column halves are kHalfKV apart,
// 8-key groups 1024 bytes apart.
__device__ __forceinline__ uint64_t desc_v(uint32_t saddr) { return smem_desc(saddr, kHalfKV, 1024); }

struct Bars {
  uint64_t q_full, q_empty;
  uint64_t k_full[kStages], v_full[kStages], kv_empty[kStages];
  uint64_t s_full[2], s_free[2], p_full[2], pv_done[2];
  uint64_t o_full, o_empty;
};
static_assert(sizeof(Bars) == kNumBars * 8, "barrier block");
static_assert(kSmem <= 232448, "shared memory");

__global__ void __launch_bounds__(kThreads, 1) mma_attn_kernel(const AttnParams p,
                                                               const __grid_constant__ CUtensorMap qmap,
                                                               const __grid_constant__ CUtensorMap kmap,
                                                               const __grid_constant__ CUtensorMap vmap) {
  extern __shared__ __align__(1024) uint8_t smem[];
  if (smem_u32(smem) & 1023u) {  // uniform: every thread returns before any barrier
    if (threadIdx.x == 0) raise_error(p.err, PKV_DEVERR_INTERNAL);
    return;
  }
  Bars* bars = reinterpret_cast<Bars*>(smem + kBarOff);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kBarOff + kNumBars * 8);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(&bars->q_full, 1);
    mbar_init(&bars->q_empty, 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bars->k_full[s], 1);
      mbar_init(&bars->v_full[s], 1);
      mbar_init(&bars->kv_empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bars->s_full[b], 1);
      mbar_init(&bars->s_free[b], 256);
      mbar_init(&bars->p_full[b], 256);
      mbar_init(&bars->pv_done[b], 1);
    }
    mbar_init(&bars->o_full, 1);
    mbar_init(&bars->o_empty, 256);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  pdl_wait();  // the plan and the K/V write are complete and visible from here on
  const int n_items = p.header->n_mma;
  const uint32_t tmem = *tmem_slot;
  const uint32_t smem_base = smem_u32(smem);

  // One counter g numbers the key tiles this CTA processes (across items):
  // ring stage g % kStages (parity (g / kStages) & 1), S and P buffer g & 1
  // (parity (g >> 1) & 1).
  if (warp == 0) {
    // ================================================================ producer
    if (lane == 0) {
      prefetch_tensormap(&qmap);
      prefetch_tensormap(&kmap);
      prefetch_tensormap(&vmap);
    }
    const int nb = kKeys / p.bs;
    int g = 0, it_cnt = 0;
    bool ok = true;
    for (int idx = blockIdx.x; idx < n_items && ok; idx += gridDim.x, ++it_cnt) {
      const WorkItem it = p.items[idx];
      const int L = p.context_lens[it.seq];
      const int qstart = p.query_start_loc[it.seq];
      const int nblk = (L + p.bs - 1) / p.bs;
      const int32_t* bt = p.block_tables + (int64_t)it.seq * p.max_blocks;
      auto block_of = [&](int kbase) -> int {  // physical block of this lane's block in the tile
        const int lb = kbase / p.bs + lane;
        int phys = (int)p.num_blocks;  // out of range: reads as zeros
        if (lane < nb && lb < nblk) {
          const int b = __ldg(bt + lb);
          if (b >= 0 && (int64_t)b < p.num_blocks)
            phys = b;
          else
            raise_error(p.err, PKV_DEVERR_BLOCK_OUT_OF_RANGE);
        }
        return phys;
      };
      int phys = block_of(it.kb);
      // Q tile: reusable once the previous item's last S MMA has completed
      if (!__all_sync(0xffffffffu, mbar_wait(&bars->q_empty, (it_cnt & 1) ^ 1, p.err))) break;
      if (lane == 0) {
        mbar_arrive_expect_tx(&bars->q_full, kQBytes);
        const int tok0 = qstart + it.row0 / p.G;
        tma_load_3d(smem + kQOff, &qmap, &bars->q_full, 0, it.kvh * p.G, tok0);
        tma_load_3d(smem + kQOff + kHalf, &qmap, &bars->q_full, 64, it.kvh * p.G, tok0);
      }
      for (int kbase = it.kb; kbase < it.ke; kbase += kKeys, ++g) {
        const int st = g % kStages;
        const int next_phys = (kbase + kKeys < it.ke) ? block_of(kbase + kKeys) : 0;
        if (!__all_sync(0xffffffffu, mbar_wait(&bars->kv_empty[st], ((g / kStages) & 1) ^ 1, p.err))) {
          ok = false;
          break;
        }
        if (lane == 0) {
          mbar_arrive_expect_tx(&bars->k_full[st], kTileBytes);
          mbar_arrive_expect_tx(&bars->v_full[st], kTileBytes);
        }
        __syncwarp();
        if (lane < nb) {
          const int row_off = lane * p.bs * 128;
          uint8_t* kd = smem + kSOff + st * kStageBytes + row_off;
          uint8_t* vd = kd + kTileBytes;
          tma_load_4d(kd, &kmap, &bars->k_full[st], 0, it.kvh, 0, phys);
          tma_load_4d(kd + kHalfKV, &kmap, &bars->k_full[st], 64, it.kvh, 0, phys);
          tma_load_4d(vd, &vmap, &bars->v_full[st], 0, it.kvh, 0, phys);
          tma_load_4d(vd + kHalfKV, &vmap, &bars->v_full[st], 64, it.kvh, 0, phys);
        }
        phys = next_phys;
      }
    }
  } else if (warp == 1) {
    // ================================================================ MMA issuer
    if (lane == 0) {
      int g = 0, it_cnt = 0;
      bool ok = true;
      // O (+)= P V for tile gp; `first` starts the item's accumulation.
      auto issue_pv = [&](int gp, bool first) -> bool {
        const int b = gp & 1, st = gp % kStages;
        if (!mbar_wait(&bars->p_full[b], (gp >> 1) & 1, p.err)) return false;
        if (!mbar_wait(&bars->v_full[st], (gp / kStages) & 1, p.err)) return false;
        tc_fence_after();
        const uint32_t pbase = smem_base + kPOff + b * kPBytes;
        const uint32_t vbase = smem_base + kSOff + st * kStageBytes + kTileBytes;
#pragma unroll
        for (int kk = 0; kk < kKeys / 16; ++kk)
          umma_bf16(tmem + kOCol, desc_k(pbase + kk * 32), desc_v(vbase + kk * 2048), kIdescO,
                    (first && kk == 0) ? 0u : 1u);
        umma_commit(&bars->pv_done[b]);
        umma_commit(&bars->kv_empty[st]);
        return true;
      };
      for (int idx = blockIdx.x; idx < n_items && ok; idx += gridDim.x, ++it_cnt) {
        const WorkItem it = p.items[idx];
        if (!mbar_wait(&bars->q_full, it_cnt & 1, p.err)) break;
        const int ntiles = (it.ke - it.kb + kKeys - 1) / kKeys;
        for (int j = 0; j < ntiles; ++j, ++g) {
          const int b = g & 1, st = g % kStages;
          if (!mbar_wait(&bars->k_full[st], (g / kStages) & 1, p.err) ||
              !mbar_wait(&bars->s_free[b], ((g >> 1) & 1) ^ 1, p.err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t qbase = smem_base + kQOff;
          const uint32_t kbase = smem_base + kSOff + st * kStageBytes;
#pragma unroll
          for (int kk = 0; kk < 128 / 16; ++kk)
            umma_bf16(tmem + kSCol + b * kKeys, desc_k(qbase + (kk >> 2) * kHalf + (kk & 3) * 32),
                      desc_k(kbase + (kk >> 2) * kHalfKV + (kk & 3) * 32), kIdescS, kk > 0 ? 1u : 0u);
          umma_commit(&bars->s_full[b]);
          if (j == ntiles - 1) umma_commit(&bars->q_empty);  // Q no longer read by this item
          if (j == 0 && it_cnt > 0) {
            // O is about to be overwritten: the previous item's epilogue must have read it
            if (!mbar_wait(&bars->o_empty, (it_cnt - 1) & 1, p.err)) {
              ok = false;
              break;
            }
          }
          if (j > 0 && !issue_pv(g - 1, j == 1)) {
            ok = false;
            break;
          }
        }
        if (!ok) break;
        if (!issue_pv(g - 1, ntiles == 1)) break;
        umma_commit(&bars->o_full);
      }
    }
    __syncwarp();
  } else {
    // ================================================================ softmax / epilogue
    const int q4 = warp & 3;
    const int h = (warp - 2) >> 2;  // key half of a tile (columns 32h .. 32h+31); output half 64h .. 64h+63
    const int r = q4 * 32 + lane;   // row of the tile == TMEM lane
    const int pair_bar = 1 + q4;    // warps (w, w+4) of one row quarter
    const uint32_t lane_base = tmem + ((uint32_t)(q4 * 32) << 16);
    float* red = reinterpret_cast<float*>(smem + kRedOff);
    int g = 0, it_cnt = 0;
    bool ok = true;
    for (int idx = blockIdx.x; idx < n_items && ok; idx += gridDim.x, ++it_cnt) {
      const WorkItem it = p.items[idx];
      const int L = p.context_lens[it.seq];
      const int qstart = p.query_start_loc[it.seq];
      const int n = p.query_start_loc[it.seq + 1] - qstart;
      const bool valid = r < it.nrows;
      const int row = it.row0 + r;
      const int tok = row / p.G, gh = row - tok * p.G;
      const int vis = valid ? min(it.ke, p.causal ? L - n + tok + 1 : L) : 0;
      float m_ref = -CUDART_INF_F, l = 0.f;
      const int ntiles = (it.ke - it.kb + kKeys - 1) / kKeys;
      for (int j = 0; j < ntiles; ++j, ++g) {
        const int b = g & 1, st = g % kStages;
        const int kt = it.kb + j * kKeys;  // first key of the tile
        if (!__all_sync(0xffffffffu, mbar_wait(&bars->s_full[b], (g >> 1) & 1, p.err))) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t sraw[32];
        tmem_ld32(lane_base + kSCol + b * kKeys + 32 * h, sraw);
        tmem_wait_ld();
        tc_fence_before();
        mbar_arrive(&bars->s_free[b]);
        const int nvis = vis - (kt + 32 * h);  // keys c < nvis of this half are visible
        if (nvis < 32) {
#pragma unroll
          for (int c = 0; c < 32; ++c)
            if (c >= nvis) sraw[c] = __float_as_uint(-CUDART_INF_F);
        }
        float m4[4] = {-CUDART_INF_F, -CUDART_INF_F, -CUDART_INF_F, -CUDART_INF_F};
#pragma unroll
        for (int c = 0; c < 32; ++c) m4[c & 3] = fmaxf(m4[c & 3], __uint_as_float(sraw[c]));
        float mx = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
        float* redm = red + b * 256;
        redm[h * 128 + r] = mx;
        named_barrier(pair_bar, 64);
        mx = fmaxf(mx, redm[(h ^ 1) * 128 + r]) * p.scale_log2;
        float alpha = 1.f;
        bool rescale = false;
        if (mx > m_ref + kRescaleThreshold) {  // false while both are -inf
          alpha = fast_exp2(m_ref - mx);       // 0 when m_ref is -inf
          rescale = j > 0 && m_ref != -CUDART_INF_F;
          m_ref = mx;
        }
        const float neg_m = m_ref == -CUDART_INF_F ? 0.f : -m_ref;
        // P buffer b is free once the P.V that read it two tiles ago is done
        if (!__all_sync(0xffffffffu, mbar_wait(&bars->pv_done[b], ((g >> 1) & 1) ^ 1, p.err))) {
          ok = false;
          break;
        }
        uint8_t* prow = smem + kPOff + b * kPBytes + r * 128;
        float ps[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int u = 0; u < 4; ++u) {  // 16-byte chunks of 8 keys: chunk 4h + u of the row
          float e[8];
#pragma unroll
          for (int t = 0; t < 8; ++t) {
            e[t] = fast_exp2(fmaf(__uint_as_float(sraw[u * 8 + t]), p.scale_log2, neg_m));
            ps[t & 3] += e[t];
          }
          uint4 w;
          w.x = pack_bf16(e[0], e[1]);
          w.y = pack_bf16(e[2], e[3]);
          w.z = pack_bf16(e[4], e[5]);
          w.w = pack_bf16(e[6], e[7]);
          *reinterpret_cast<uint4*>(prow + (((4 * h + u) ^ (r & 7)) << 4)) = w;
        }
        l = fmaf(l, alpha, (ps[0] + ps[1]) + (ps[2] + ps[3]));
        if (__any_sync(0xffffffffu, rescale)) {
          // O must hold every earlier tile's P.V before it is scaled; the TMEM
          // accesses are warp-wide, rows that keep their max scale by 1
          if (!__all_sync(0xffffffffu, mbar_wait(&bars->pv_done[b ^ 1], ((g - 1) >> 1) & 1, p.err))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const float f = rescale ? alpha : 1.f;
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            uint32_t o[32];
            tmem_ld32(lane_base + kOCol + 64 * h + c * 32, o);
            tmem_wait_ld();
#pragma unroll
            for (int t = 0; t < 32; ++t) o[t] = __float_as_uint(__uint_as_float(o[t]) * f);
            tmem_st32(lane_base + kOCol + 64 * h + c * 32, o);
          }
          tmem_wait_st();
        }
        if (kt + kKeys > L) {
          // keys at or past the sequence's end hold arbitrary bits: zero their V
          // rows (thread: key r of the tile, d-half h) so that 0 * V stays 0
          if (!__all_sync(0xffffffffu, mbar_wait(&bars->v_full[st], (g / kStages) & 1, p.err))) {
            ok = false;
            break;
          }
          if (r < kKeys && kt + r >= L) {
            uint4* v0 =
                reinterpret_cast<uint4*>(smem + kSOff + st * kStageBytes + kTileBytes + h * kHalfKV + r * 128);
#pragma unroll
            for (int t = 0; t < 8; ++t) v0[t] = make_uint4(0, 0, 0, 0);
          }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(&bars->p_full[b]);
      }
      if (!ok) break;
      // ---- epilogue: row sum of the pair, O (this thread's 64 output columns) / l.
      // The sums go through the max buffer the last tile did not use; the
      // second pair barrier keeps the next tile from overwriting them early.
      float* reds = red + (g & 1) * 256;
      reds[h * 128 + r] = l;
      named_barrier(pair_bar, 64);
      const float ltot = l + reds[(h ^ 1) * 128 + r];
      named_barrier(pair_bar, 64);
      if (!__all_sync(0xffffffffu, mbar_wait(&bars->o_full, it_cnt & 1, p.err))) break;
      tc_fence_after();
      uint32_t o[64];
      tmem_ld32(lane_base + kOCol + 64 * h, o);
      tmem_ld32(lane_base + kOCol + 64 * h + 32, o + 32);
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive(&bars->o_empty);
      if (valid) {
        if (it.part < 0) {
          const float inv = 1.f / ltot;
          __nv_bfloat16* orow = reinterpret_cast<__nv_bfloat16*>(p.out) +
                                ((int64_t)(qstart + tok) * p.Hq + (int64_t)it.kvh * p.G + gh) * 128 + 64 * h;
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            uint4 w;
            w.x = pack_bf16(__uint_as_float(o[u * 8 + 0]) * inv, __uint_as_float(o[u * 8 + 1]) * inv);
            w.y = pack_bf16(__uint_as_float(o[u * 8 + 2]) * inv, __uint_as_float(o[u * 8 + 3]) * inv);
            w.z = pack_bf16(__uint_as_float(o[u * 8 + 4]) * inv, __uint_as_float(o[u * 8 + 5]) * inv);
            w.w = pack_bf16(__uint_as_float(o[u * 8 + 6]) * inv, __uint_as_float(o[u * 8 + 7]) * inv);
            *reinterpret_cast<uint4*>(orow + u * 8) = w;
          }
        } else {
          float4* dst = reinterpret_cast<float4*>(p.part_acc + (int64_t)(it.part + r) * 128 + 64 * h);
#pragma unroll
          for (int u = 0; u < 16; ++u)
            dst[u] = make_float4(__uint_as_float(o[u * 4]), __uint_as_float(o[u * 4 + 1]),
                                 __uint_as_float(o[u * 4 + 2]), __uint_as_float(o[u * 4 + 3]));
          if (h == 0) p.part_ml[it.part + r] = make_float2(m_ref, ltot);
        }
      }
      if (it.part >= 0) {
        // The split that completes its merge group combines the group's
        // partial rows: m = max m_p, l = sum l_p 2^(m_p - m), O = sum acc_p 2^(m_p - m) / l.
        // Release: the barrier orders every thread's partial writes before one
        // thread's fence and ticket; acquire: that thread's fence, then the barrier.
        int* flag_last = reinterpret_cast<int*>(tmem_slot + 1);
        named_barrier(5, 256);
        if (r == 0 && h == 0) {
          __threadfence();
          *flag_last = atomicAdd(p.tickets + it.grp, 1);
        }
        named_barrier(5, 256);
        const MergeGroup gr = p.groups[it.grp];
        if (*flag_last == gr.nsplit - 1) {
          if (r == 0 && h == 0) __threadfence();
          named_barrier(5, 256);
          if (r < gr.nrows) {
            float M = -CUDART_INF_F;
#pragma unroll 8
            for (int sp = 0; sp < gr.nsplit; ++sp)
              M = fmaxf(M, __ldcg(&p.part_ml[gr.part_base + sp * gr.nrows + r]).x);
            const float Mu = M == -CUDART_INF_F ? 0.f : M;
            float lsum = 0.f;
            float acc[64];
#pragma unroll
            for (int c = 0; c < 64; ++c) acc[c] = 0.f;
            for (int sp = 0; sp < gr.nsplit; ++sp) {
              const int slot = gr.part_base + sp * gr.nrows + r;
              const float2 ml = __ldcg(&p.part_ml[slot]);
              const float wt = fast_exp2(ml.x - Mu);
              lsum = fmaf(wt, ml.y, lsum);
              const float4* src = reinterpret_cast<const float4*>(p.part_acc + (int64_t)slot * 128 + 64 * h);
#pragma unroll
              for (int u = 0; u < 16; ++u) {
                const float4 a = __ldcg(src + u);
                acc[4 * u] = fmaf(wt, a.x, acc[4 * u]);
                acc[4 * u + 1] = fmaf(wt, a.y, acc[4 * u + 1]);
                acc[4 * u + 2] = fmaf(wt, a.z, acc[4 * u + 2]);
                acc[4 * u + 3] = fmaf(wt, a.w, acc[4 * u + 3]);
              }
            }
            const float inv = 1.f / lsum;
            const int grow = gr.row0 + r;
            const int gtok = grow / p.G, ggh = grow - gtok * p.G;
            __nv_bfloat16* orow = reinterpret_cast<__nv_bfloat16*>(p.out) +
                                  ((int64_t)(qstart + gtok) * p.Hq + (int64_t)gr.kvh * p.G + ggh) * 128 + 64 * h;
#pragma unroll
            for (int u = 0; u < 8; ++u) {
              uint4 w;
              w.x = pack_bf16(acc[u * 8 + 0] * inv, acc[u * 8 + 1] * inv);
              w.y = pack_bf16(acc[u * 8 + 2] * inv, acc[u * 8 + 3] * inv);
              w.z = pack_bf16(acc[u * 8 + 4] * inv, acc[u * 8 + 5] * inv);
              w.w = pack_bf16(acc[u * 8 + 6] * inv, acc[u * 8 + 7] * inv);
              *reinterpret_cast<uint4*>(orow + u * 8) = w;
            }
          }
        }
        named_barrier(5, 256);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

}  // namespace

cudaError_t launch_mma(const AttnParams& p, const CUtensorMap& qmap, const CUtensorMap& kmap, const CUtensorMap& vmap,
                       int grid, cudaStream_t s) {
  static unsigned long long done_mask = 0;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!(__atomic_load_n(&done_mask, __ATOMIC_ACQUIRE) & (1ull << dev))) {
    e = cudaFuncSetAttribute(mma_attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e != cudaSuccess) return e;
    __atomic_fetch_or(&done_mask, 1ull << dev, __ATOMIC_RELEASE);
  }
  e = launch_pdl(mma_attn_kernel, dim3(grid), dim3(kThreads), kSmem, s, p, qmap, kmap, vmap);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace pkv
