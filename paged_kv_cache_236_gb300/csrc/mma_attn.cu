// Tensor-core paged attention for multi-token queries (prefill chunks,
// speculative verification): tcgen05.mma with TMEM accumulators.
//
// What it computes is the same as the CUDA-core kernel ("Paged Attention
// 基础", section 2, steps 1-5; causal mask at each query's absolute position
// L - n + i, "ADR 004" Consequences: prefill and decode share one call), for
// a work item of up to 128 rows (query token, head-in-group) of one sequence
// and one kv head over keys [kb, ke):
//   S = Q K^T (128 x 128 per key tile, fp32 in TMEM), online softmax in
//   registers (one thread per row), P (bf16) -> shared memory, O += P V
//   (fp32 in TMEM), O / l at the end (or a partial (m, l, O) row for split-KV).
//
// Roles (192 threads, one CTA per SM, persistent over items):
//   warp 0    TMA producer: the item's Q tile (3-D box {64, G heads, 128/G
//             tokens} of q [T, Hq, D], two 64-column halves) and, per
//             128-key tile, one {64, 1, block_size, 1} box per physical block
//             and half of the pool [NB, bs, Hkv, D] for K and for V
//             (128-byte swizzle, the layout the tensor core reads);
//   warp 1    TMEM allocation and the single thread that issues the MMAs;
//   warps 2-5 softmax / correction / epilogue, thread i of the 128 owning
//             TMEM lane (row) 32*(warp%4) + i.
// Shared memory: Q 32 KB, 2 stages of K+V (128 KB), 2 P buffers (64 KB).
// TMEM: S double-buffered in columns [0,256), O in [256,384).
//
// The running max used for the exponentials is only raised when a tile's row
// maximum exceeds it by more than 8 (log2 units), so O is rescaled in TMEM
// rarely; P stays <= 2^8 and the result is exact up to rounding.
#include <math_constants.h>

#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace {

constexpr int kThreads = 192;
constexpr int kStages = 2;
constexpr int kTileBytes = kMmaTileKeys * 128 * 2;  // 128 keys x 128 dims x bf16 = 32 KB
constexpr int kQBytes = kMmaRows * 128 * 2;          // 32 KB
constexpr int kPBytes = kMmaRows * kMmaTileKeys * 2;  // 32 KB
constexpr int kHalf = 128 * 128;                      // one 64-column half of a 128-row tile (16 KB)
// shared-memory carve-up (offsets from a 1024-byte aligned base)
constexpr int kQOff = 0;
constexpr int kKOff = kQOff + kQBytes;
constexpr int kVOff = kKOff + kStages * kTileBytes;
constexpr int kPOff = kVOff + kStages * kTileBytes;
constexpr int kBarOff = kPOff + 2 * kPBytes;
constexpr int kNumBars = 2 + 3 * kStages + 2 * 4 + 2;
constexpr int kSmem = kBarOff + kNumBars * 8 + 16 + 1024;
constexpr uint32_t kTmemCols = 512;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

// ---------------------------------------------------------------------------
// tcgen05 / TMEM wrappers
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t* dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst)), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// D[tmem] (+)= A[smem] * B[smem], bf16 inputs, fp32 accumulate.
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive on `bar` once every MMA issued so far by this thread has completed.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

#define PKV_R32(i) "=r"(v[i])
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t* v) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : PKV_R32(0), PKV_R32(1), PKV_R32(2), PKV_R32(3), PKV_R32(4), PKV_R32(5), PKV_R32(6), PKV_R32(7), PKV_R32(8),
        PKV_R32(9), PKV_R32(10), PKV_R32(11), PKV_R32(12), PKV_R32(13), PKV_R32(14), PKV_R32(15), PKV_R32(16),
        PKV_R32(17), PKV_R32(18), PKV_R32(19), PKV_R32(20), PKV_R32(21), PKV_R32(22), PKV_R32(23), PKV_R32(24),
        PKV_R32(25), PKV_R32(26), PKV_R32(27), PKV_R32(28), PKV_R32(29), PKV_R32(30), PKV_R32(31)
      : "r"(taddr));
}
#undef PKV_R32
#define PKV_W32(i) "r"(v[i])
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t* v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
      PKV_W32(0), PKV_W32(1), PKV_W32(2), PKV_W32(3), PKV_W32(4), PKV_W32(5), PKV_W32(6), PKV_W32(7), PKV_W32(8),
      PKV_W32(9), PKV_W32(10), PKV_W32(11), PKV_W32(12), PKV_W32(13), PKV_W32(14), PKV_W32(15), PKV_W32(16),
      PKV_W32(17), PKV_W32(18), PKV_W32(19), PKV_W32(20), PKV_W32(21), PKV_W32(22), PKV_W32(23), PKV_W32(24),
      PKV_W32(25), PKV_W32(26), PKV_W32(27), PKV_W32(28), PKV_W32(29), PKV_W32(30), PKV_W32(31)
      : "memory");
}
#undef PKV_W32
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Shared-memory matrix descriptors (sm_100 format: start>>4 in [0,14), leading
// byte offset>>4 in [16,30), stride byte offset>>4 in [32,46), version 1 at
// [46,48), layout type at [61,64) with 2 = 128-byte swizzle).
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)((lbo_bytes >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo_bytes >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}
// K-major operand, 128-byte rows swizzled, 8-row groups 1024 bytes apart
// (Q, K, P).  The leading byte offset is not used by this layout.
__device__ __forceinline__ uint64_t desc_k(uint32_t saddr) { return smem_desc(saddr, 16, 1024); }
// MN-major operand (V as the B of P.V): 64-element halves 16 KB apart
// (leading byte offset), 8-key groups 1024 bytes apart (stride byte offset).
__device__ __forceinline__ uint64_t desc_mn(uint32_t saddr) { return smem_desc(saddr, kHalf, 1024); }

// Instruction descriptor, kind::f16: D f32 (bits 4-5 = 1), A and B bf16
// (bits 7-9 and 10-12 = 1), B major-ness at bit 16, N>>3 at 17-22, M>>4 at 24-28.
constexpr uint32_t idesc_bf16(int M, int N, bool b_mn_major) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((b_mn_major ? 1u : 0u) << 16) | ((uint32_t)(N >> 3) << 17) |
         ((uint32_t)(M >> 4) << 24);
}
constexpr uint32_t kIdescS = idesc_bf16(128, 128, false);
constexpr uint32_t kIdescO = idesc_bf16(128, 128, true);

struct Bars {
  uint64_t q_full, q_empty;
  uint64_t k_full[kStages], v_full[kStages], kv_empty[kStages];
  uint64_t s_full[2], s_free[2], p_full[2], pv_done[2];
  uint64_t o_full, o_empty;
};
static_assert(sizeof(Bars) == kNumBars * 8, "barrier block");

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&h);
}

__global__ void __launch_bounds__(kThreads, 1) mma_attn_kernel(const AttnParams p,
                                                               const __grid_constant__ CUtensorMap qmap,
                                                               const __grid_constant__ CUtensorMap kmap,
                                                               const __grid_constant__ CUtensorMap vmap) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  Bars* bars = reinterpret_cast<Bars*>(smem + kBarOff);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kBarOff + kNumBars * 8);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_items = p.header->n_mma;

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
      mbar_init(&bars->s_free[b], 128);
      mbar_init(&bars->p_full[b], 128);
      mbar_init(&bars->pv_done[b], 1);
    }
    mbar_init(&bars->o_full, 1);
    mbar_init(&bars->o_empty, 128);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t smem_base = smem_u32(smem);

  // One counter g numbers the key tiles this CTA processes (across items);
  // stage, S buffer and P buffer of tile g are all g & 1, and the phase
  // parity of its barriers is (g >> 1) & 1.
  static_assert(kStages == 2, "stage, S buffer and P buffer share one index");
  if (warp == 0) {
    // ================================================================ producer
    if (lane == 0) {
      prefetch_tensormap(&qmap);
      prefetch_tensormap(&kmap);
      prefetch_tensormap(&vmap);
    }
    const int nb = kMmaTileKeys / p.bs;
    int g = 0, it_cnt = 0;
    bool ok = true;
    for (int idx = blockIdx.x; idx < n_items && ok; idx += gridDim.x, ++it_cnt) {
      const WorkItem it = p.items[idx];
      const int L = p.context_lens[it.seq];
      const int qstart = p.query_start_loc[it.seq];
      const int nblk = (L + p.bs - 1) / p.bs;
      const int32_t* bt = p.block_tables + (int64_t)it.seq * p.max_blocks;
      // Q tile: reusable once the previous item's last S MMA has completed
      if (!__all_sync(0xffffffffu, mbar_wait(&bars->q_empty, (it_cnt & 1) ^ 1, p.err))) break;
      if (lane == 0) {
        mbar_arrive_expect_tx(&bars->q_full, kQBytes);
        const int tok0 = qstart + it.row0 / p.G;
        tma_load_3d(smem + kQOff, &qmap, &bars->q_full, 0, it.kvh * p.G, tok0);
        tma_load_3d(smem + kQOff + kHalf, &qmap, &bars->q_full, 64, it.kvh * p.G, tok0);
      }
      for (int kbase = it.kb; kbase < it.ke; kbase += kMmaTileKeys, ++g) {
        const int st = g & 1;
        if (!__all_sync(0xffffffffu, mbar_wait(&bars->kv_empty[st], ((g >> 1) & 1) ^ 1, p.err))) {
          ok = false;
          break;
        }
        if (lane == 0) {
          mbar_arrive_expect_tx(&bars->k_full[st], kTileBytes);
          mbar_arrive_expect_tx(&bars->v_full[st], kTileBytes);
        }
        __syncwarp();
        if (lane < nb) {
          const int lb = kbase / p.bs + lane;
          int phys = (int)p.num_blocks;  // out of range: reads as zeros
          if (lb < nblk) {
            const int b = bt[lb];
            if (b >= 0 && (int64_t)b < p.num_blocks)
              phys = b;
            else
              raise_error(p.err, PKV_DEVERR_BLOCK_OUT_OF_RANGE);
          }
          const int row_off = lane * p.bs * 128;
          uint8_t* kd = smem + kKOff + st * kTileBytes + row_off;
          uint8_t* vd = smem + kVOff + st * kTileBytes + row_off;
          tma_load_4d(kd, &kmap, &bars->k_full[st], 0, it.kvh, 0, phys);
          tma_load_4d(kd + kHalf, &kmap, &bars->k_full[st], 64, it.kvh, 0, phys);
          tma_load_4d(vd, &vmap, &bars->v_full[st], 0, it.kvh, 0, phys);
          tma_load_4d(vd + kHalf, &vmap, &bars->v_full[st], 64, it.kvh, 0, phys);
        }
      }
    }
  } else if (warp == 1) {
    // ================================================================ MMA issuer
    if (lane == 0) {
      int g = 0, it_cnt = 0;
      bool ok = true;
      // O (+)= P V for tile gp; `first` starts the item's accumulation.
      auto issue_pv = [&](int gp, bool first) -> bool {
        const int b = gp & 1;
        if (!mbar_wait(&bars->p_full[b], (gp >> 1) & 1, p.err)) return false;
        if (!mbar_wait(&bars->v_full[b], (gp >> 1) & 1, p.err)) return false;
        tc_fence_after();
        const uint32_t pbase = smem_base + kPOff + b * kPBytes;
        const uint32_t vbase = smem_base + kVOff + b * kTileBytes;
#pragma unroll
        for (int kk = 0; kk < kMmaTileKeys / 16; ++kk) {
          const uint64_t a = desc_k(pbase + (kk >> 2) * kHalf + (kk & 3) * 32);
          const uint64_t bd = desc_mn(vbase + kk * 2048);
          umma_bf16(tmem + 256, a, bd, kIdescO, (first && kk == 0) ? 0u : 1u);
        }
        umma_commit(&bars->pv_done[b]);
        umma_commit(&bars->kv_empty[b]);
        return true;
      };
      for (int idx = blockIdx.x; idx < n_items && ok; idx += gridDim.x, ++it_cnt) {
        const WorkItem it = p.items[idx];
        if (!mbar_wait(&bars->q_full, it_cnt & 1, p.err)) break;
        const int ntiles = (it.ke - it.kb + kMmaTileKeys - 1) / kMmaTileKeys;
        for (int j = 0; j < ntiles; ++j, ++g) {
          const int b = g & 1;
          if (!mbar_wait(&bars->k_full[b], (g >> 1) & 1, p.err) ||
              !mbar_wait(&bars->s_free[b], ((g >> 1) & 1) ^ 1, p.err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t qbase = smem_base + kQOff;
          const uint32_t kbase = smem_base + kKOff + b * kTileBytes;
#pragma unroll
          for (int kk = 0; kk < 128 / 16; ++kk) {
            const uint32_t off = (kk >> 2) * kHalf + (kk & 3) * 32;
            umma_bf16(tmem + b * 128, desc_k(qbase + off), desc_k(kbase + off), kIdescS, kk > 0 ? 1u : 0u);
          }
          umma_commit(&bars->s_full[b]);
          if (j == ntiles - 1) umma_commit(&bars->q_empty);  // Q no longer read by this item
          if (j == 0 && it_cnt > 0) {
            // O is about to be overwritten: the previous item's epilogue must have read it
            if (!mbar_wait(&bars->o_empty, ((it_cnt - 1) & 1), p.err)) {
              ok = false;
              break;
            }
          }
          // P.V of the previous tile goes after this tile's S so that the
          // softmax of this tile overlaps the tensor core
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
    const int r = q4 * 32 + lane;  // row of the tile == TMEM lane
    const uint32_t lane_base = tmem + ((uint32_t)(q4 * 32) << 16);
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
      const int ntiles = (it.ke - it.kb + kMmaTileKeys - 1) / kMmaTileKeys;
      for (int j = 0; j < ntiles; ++j, ++g) {
        const int b = g & 1;
        const int k0 = it.kb + j * kMmaTileKeys;
        if (!__all_sync(0xffffffffu, mbar_wait(&bars->s_full[b], (g >> 1) & 1, p.err))) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t sraw[128];
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld32(lane_base + b * 128 + c * 32, sraw + c * 32);
        tmem_wait_ld();
        tc_fence_before();
        mbar_arrive(&bars->s_free[b]);
        // scale, mask, row max
        const int nvis = vis - k0;  // keys c < nvis of this tile are visible
        float mx = -CUDART_INF_F;
#pragma unroll
        for (int c = 0; c < 128; ++c) {
          const float s = c < nvis ? __uint_as_float(sraw[c]) * p.scale_log2 : -CUDART_INF_F;
          sraw[c] = __float_as_uint(s);
          mx = fmaxf(mx, s);
        }
        float alpha = 1.f;
        bool rescale = false;
        if (mx > m_ref + kRescaleThreshold) {  // false while both are -inf
          alpha = exp2f(m_ref - mx);           // 0 when m_ref is -inf
          rescale = j > 0 && m_ref != -CUDART_INF_F;
          m_ref = mx;
        }
        const float m_use = m_ref == -CUDART_INF_F ? 0.f : m_ref;
        // P buffer b is free once the P.V that read it two tiles ago is done
        if (!__all_sync(0xffffffffu, mbar_wait(&bars->pv_done[b], ((g >> 1) & 1) ^ 1, p.err))) {
          ok = false;
          break;
        }
        uint8_t* prow = smem + kPOff + b * kPBytes + r * 128;
        float psum = 0.f;
#pragma unroll
        for (int u = 0; u < 16; ++u) {  // 16-byte chunks of 8 keys
          float e[8];
#pragma unroll
          for (int t = 0; t < 8; ++t) {
            e[t] = exp2f(__uint_as_float(sraw[u * 8 + t]) - m_use);
            psum += e[t];
          }
          uint4 w;
          w.x = pack_bf16(e[0], e[1]);
          w.y = pack_bf16(e[2], e[3]);
          w.z = pack_bf16(e[4], e[5]);
          w.w = pack_bf16(e[6], e[7]);
          const int half = u >> 3, cu = u & 7;
          *reinterpret_cast<uint4*>(prow + half * kHalf + ((cu ^ (r & 7)) << 4)) = w;
        }
        l = l * alpha + psum;
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
          for (int c = 0; c < 4; ++c) {
            uint32_t o[32];
            tmem_ld32(lane_base + 256 + c * 32, o);
            tmem_wait_ld();
#pragma unroll
            for (int t = 0; t < 32; ++t) o[t] = __float_as_uint(__uint_as_float(o[t]) * f);
            tmem_st32(lane_base + 256 + c * 32, o);
          }
          tmem_wait_st();
        }
        if (k0 + kMmaTileKeys > L) {
          // keys at or past the sequence's end hold arbitrary bits: zero their V
          // rows (after the tile has landed) so that 0 * V stays 0
          if (!__all_sync(0xffffffffu, mbar_wait(&bars->v_full[b], (g >> 1) & 1, p.err))) {
            ok = false;
            break;
          }
          if (k0 + r >= L) {
            uint4* v0 = reinterpret_cast<uint4*>(smem + kVOff + b * kTileBytes + r * 128);
            uint4* v1 = reinterpret_cast<uint4*>(smem + kVOff + b * kTileBytes + kHalf + r * 128);
#pragma unroll
            for (int t = 0; t < 8; ++t) v0[t] = v1[t] = make_uint4(0, 0, 0, 0);
          }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(&bars->p_full[b]);
      }
      if (!ok) break;
      // ---- epilogue
      if (!__all_sync(0xffffffffu, mbar_wait(&bars->o_full, it_cnt & 1, p.err))) break;
      tc_fence_after();
      uint32_t o[128];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld32(lane_base + 256 + c * 32, o + c * 32);
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive(&bars->o_empty);
      if (valid) {
        if (it.part < 0) {
          const float inv = 1.f / l;
          __nv_bfloat16* orow = reinterpret_cast<__nv_bfloat16*>(p.out) +
                                ((int64_t)(qstart + tok) * p.Hq + (int64_t)it.kvh * p.G + gh) * 128;
#pragma unroll
          for (int u = 0; u < 16; ++u) {
            uint4 w;
            w.x = pack_bf16(__uint_as_float(o[u * 8 + 0]) * inv, __uint_as_float(o[u * 8 + 1]) * inv);
            w.y = pack_bf16(__uint_as_float(o[u * 8 + 2]) * inv, __uint_as_float(o[u * 8 + 3]) * inv);
            w.z = pack_bf16(__uint_as_float(o[u * 8 + 4]) * inv, __uint_as_float(o[u * 8 + 5]) * inv);
            w.w = pack_bf16(__uint_as_float(o[u * 8 + 6]) * inv, __uint_as_float(o[u * 8 + 7]) * inv);
            *reinterpret_cast<uint4*>(orow + u * 8) = w;
          }
        } else {
          float4* dst = reinterpret_cast<float4*>(p.part_acc + (int64_t)(it.part + r) * 128);
#pragma unroll
          for (int u = 0; u < 32; ++u)
            dst[u] = make_float4(__uint_as_float(o[u * 4]), __uint_as_float(o[u * 4 + 1]),
                                 __uint_as_float(o[u * 4 + 2]), __uint_as_float(o[u * 4 + 3]));
          p.part_ml[it.part + r] = make_float2(m_ref, l);
        }
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
  mma_attn_kernel<<<grid, kThreads, kSmem, s>>>(p, qmap, kmap, vmap);
  return cudaGetLastError();
}

}  // namespace pkv
