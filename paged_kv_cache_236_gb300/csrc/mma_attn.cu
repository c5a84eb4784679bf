// Tensor-core paged attention for multi-token queries (prefill chunks,
// speculative verification): tcgen05.mma with TMEM accumulators.
//
// What it computes is the same as the other attention kernels ("Paged
// Attention 基础", section 2, steps 1-5; causal mask at each query's absolute
// position L - n + i; "ADR 004" Consequences: prefill and decode share one
// call), for a work item of up to 128 rows (query token, head-in-group) of one
// sequence and one kv head over keys [kb, ke):
//   S = Q K^T (128 rows x 128 keys per tile, fp32 in TMEM), online softmax in
//   registers, P (bf16) written to TMEM, O += P V (fp32 in TMEM; the tensor
//   core reads P from TMEM and V from shared memory), O / l at the end, or a
//   partial (m, l, O) row for split-KV; the last split of a merge group to
//   finish merges the group (atomic ticket, no waiting).
//
// Tile shape and issue order follow the tensor pipe's behaviour on sm_103a:
// an M=128 MMA with N=64 costs about as long as one with N=128; a chain of
// MMAs accumulating into one TMEM region runs at about two thirds of the peak
// rate alone, at the peak when a second, independent chain runs beside it,
// whether one thread or two issue them; and one thread cannot issue faster
// than the pipe runs, so every wait or commit between its MMAs leaves the
// pipe idle.  So a tile is 128 keys (N=128 for Q K^T), and two threads issue
// the MMAs, each with its own waits: one the Q K^T chains, as soon as the
// softmax warps have read the S buffer it writes, the other the P.V chains,
// as soon as their P is written.  Either one's waits overlap the other's MMAs.
//
// Roles (384 threads, one CTA per SM, persistent; items are taken from an
// atomic counter in the planner's largest-first order, so SMs that run
// slower take fewer):
//   warp 0    the thread issuing P.V (O += P V, P from TMEM, V from shared memory);
//   warp 1    TMEM allocation and the thread issuing Q K^T (S = Q K^T);
//   warps 2-9 softmax / correction / epilogue: two threads per row (TMEM
//             lane), warps 2-5 on key columns 0-63 of a tile, warps 6-9 on
//             64-127; a pair exchanges row maxima (and at the end row sums)
//             through shared memory;
//   warp 10   item fetch, Q and K: publishes each item in a slot of shared
//             memory (with the block ids of its first key tile), loads its Q
//             tile (3-D box {64, G heads, 128/G tokens} of q [T, Hq, D], two
//             64-column halves), then its K tiles: per tile one
//             {64, 1, block_size, 1} box of the pool [NB, bs, Hkv, D] per
//             physical block and 64-column half (128-byte swizzle, the layout
//             the tensor core reads), block ids loaded a tile ahead;
//   warp 11   V producer, the same boxes from the V pool.
// Shared memory: 2 Q tiles (64 KB), a 3-stage ring of K tiles (96 KB) and a
// 2-stage ring of V tiles (64 KB); K of a tile is released when its Q K^T is
// done, V when its P.V is done (K is needed two tiles ahead of V).
// TMEM (512 columns): S double-buffered in [0,256), P (32 columns of packed
// bf16 per 64 keys) double-buffered in [256,384), O in [384,512).
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

constexpr int kThreads = 384;
constexpr int kKeys = kMmaTileKeys;                 // 128 keys per tile
constexpr int kKStages = 3, kVStages = 2;
constexpr int kHalfKV = kKeys * 128;                // one 64-column half of a K or V tile (16 KB)
constexpr int kTileBytes = 2 * kHalfKV;             // K or V tile: 32 KB
constexpr int kQBytes = kMmaRows * 128 * 2;         // 32 KB (two 16 KB halves)
// shared-memory carve-up (offsets from a 1024-byte aligned base)
constexpr int kQOff = 0;
constexpr int kKOff = kQOff + 2 * kQBytes;
constexpr int kVOff = kKOff + kKStages * kTileBytes;
constexpr int kBarOff = kVOff + kVStages * kTileBytes;
constexpr int kNumBars = 8 + 2 * kKStages + kVStages + 8 + 1;
constexpr int kSlotOff = (kBarOff + kNumBars * 8 + 16 + 15) & ~15;  // 2 item slots
constexpr int kRedOff = kSlotOff + 2 * 176;         // [2 tiles][2 halves][128 rows] row maxima / sums
// No alignment slack: the buffers need a 1024-byte aligned base, which the
// dynamic shared memory of a kernel without static shared memory has; the
// kernel checks and refuses to run otherwise.
constexpr int kSmem = kRedOff + 2 * 2 * 128 * 4;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kSCol = 0;    // S buffer b at kSCol + 128 b
constexpr uint32_t kPCol = 256;  // P buffer b at kPCol + 64 b
constexpr uint32_t kOCol = 384;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

constexpr uint32_t kIdescS = idesc_bf16(128, kKeys, false, false);
constexpr uint32_t kIdescO = idesc_bf16(128, 128, false, true);

// V as the B of P.V (MN-major): the two 64-column halves are kHalfKV apart,
// 8-key groups 1024 bytes apart.
__device__ __forceinline__ uint64_t desc_v(uint32_t saddr) { return smem_desc(saddr, kHalfKV, 1024); }

struct Bars {
  uint64_t q_full[2], q_empty[2], slot_full[2], slot_free[2];
  uint64_t k_full[kKStages], k_empty[kKStages];
  uint64_t v_full[kVStages];
  // s_full[b], phase n: S of tile 2n+b complete; s_free[b]: the softmax
  // warps have read it.  pv_done[b], phase n: the P.V of tile 2n+b complete,
  // and with it every earlier P.V.
  uint64_t s_full[2], s_free[2], pv_done[2], p_full[2];
  uint64_t o_empty;
};

// An item's description, published by the item-fetching warp before its Q
// tile is loaded (slot_full), with the block ids of its first key tile.
struct alignas(16) ItemSlot {
  WorkItem it;
  int L, qstart, n, done;
  int phys0[32];
};
// readers of a slot: the 256 softmax threads, the two MMA-issuing threads, the V producer
constexpr int kSlotReaders = 256 + 1 + 1 + 1;

static_assert(sizeof(ItemSlot) == 176, "item slot");
static_assert(sizeof(Bars) == kNumBars * 8, "barrier block");
static_assert(kVStages == 2, "V stage t % 2 is released by the P.V barrier of tile t");
static_assert(kSmem <= 232448, "shared memory");
static_assert(kKOff % 1024 == 0 && kVOff % 1024 == 0 && kTileBytes % 1024 == 0 && kQBytes % 1024 == 0,
              "swizzled tiles");
static_assert(kBarOff % 8 == 0 && kSlotOff % alignof(ItemSlot) == 0 && kRedOff % 16 == 0, "alignment");

// 64 bf16 (128 bytes) of an output row: four 32-byte stores when the output
// is 32-byte aligned, else eight 16-byte ones.
__device__ __forceinline__ void store_row128(__nv_bfloat16* dst, const uint32_t* w, int al32) {
  if (al32) {
#pragma unroll
    for (int u = 0; u < 4; ++u) st_global_v8(dst + 16 * u, w + 8 * u);
  } else {
#pragma unroll
    for (int u = 0; u < 8; ++u)
      *reinterpret_cast<uint4*>(dst + 8 * u) = make_uint4(w[4 * u], w[4 * u + 1], w[4 * u + 2], w[4 * u + 3]);
  }
}

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
  ItemSlot* slots = reinterpret_cast<ItemSlot*>(smem + kSlotOff);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bars->q_full[b], 1);
      mbar_init(&bars->q_empty[b], 1);
      mbar_init(&bars->slot_full[b], 32);
      mbar_init(&bars->slot_free[b], kSlotReaders);
      mbar_init(&bars->s_full[b], 1);
      mbar_init(&bars->s_free[b], 256);
      mbar_init(&bars->pv_done[b], 1);
      mbar_init(&bars->p_full[b], 256);
    }
    for (int s = 0; s < kKStages; ++s) {
      mbar_init(&bars->k_full[s], 1);
      mbar_init(&bars->k_empty[s], 1);
    }
    for (int s = 0; s < kVStages; ++s) mbar_init(&bars->v_full[s], 1);
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

  // One counter g numbers the key tiles this CTA processes (across items): K
  // stage g % 2 (parity (g / 2) & 1), V stage g % 3 (parity (g / 3) & 1), S
  // and P buffer g % 2.  Item c of this CTA uses Q tile and slot c & 1
  // (parity (c >> 1) & 1); O's phases count items.
  const int nb = kKeys / p.bs;  // physical blocks per tile
  // physical block of this lane's block in the tile of keys from kbase
  auto block_of = [&](const int32_t* bt, int nblk, int kbase) -> int {
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

  if (warp == 10) {
    // ================================================================ item fetch, Q and K
    if (lane == 0) {
      prefetch_tensormap(&qmap);
      prefetch_tensormap(&kmap);
    }
    int next = 0;
    if (lane == 0) next = atomicAdd(p.counter, 1);
    int g = 0;
    bool ok = true;
    for (int c = 0; ok; ++c) {
      const int qb = c & 1;
      // slot and Q tile qb: free once item c-2's last Q K^T has completed and
      // every reader has taken its description
      if (!__all_sync(0xffffffffu, mbar_wait(&bars->q_empty[qb], ((c >> 1) & 1) ^ 1, p.err) &&
                                       mbar_wait(&bars->slot_free[qb], ((c >> 1) & 1) ^ 1, p.err)))
        break;
      const int idx = __shfl_sync(0xffffffffu, next, 0);
      ItemSlot& sl = slots[qb];
      if (idx >= n_items) {
        if (lane == 0) sl.done = 1;
        mbar_arrive(&bars->slot_full[qb]);  // every lane: count 32
        if (lane == 0) mbar_arrive(&bars->q_full[qb]);
        break;
      }
      const WorkItem it = p.items[idx];
      if (lane == 0) next = atomicAdd(p.counter, 1);  // consumed at the next item
      const int L = p.context_lens[it.seq];
      const int qstart = p.query_start_loc[it.seq];
      const int nblk = (L + p.bs - 1) / p.bs;
      const int32_t* bt = p.block_tables + (int64_t)it.seq * p.max_blocks;
      int phys = block_of(bt, nblk, it.kb);
      sl.phys0[lane] = phys;
      if (lane == 0) {
        sl.it = it;
        sl.L = L;
        sl.qstart = qstart;
        sl.n = p.query_start_loc[it.seq + 1] - qstart;
        sl.done = 0;
      }
      mbar_arrive(&bars->slot_full[qb]);  // every lane, after its own writes
      if (lane == 0) {
        mbar_arrive_expect_tx(&bars->q_full[qb], kQBytes);
        const int tok0 = qstart + it.row0 / p.G;
        tma_load_3d(smem + kQOff + qb * kQBytes, &qmap, &bars->q_full[qb], 0, it.kvh * p.G, tok0);
        tma_load_3d(smem + kQOff + qb * kQBytes + kHalf, &qmap, &bars->q_full[qb], 64, it.kvh * p.G, tok0);
      }
      for (int kbase = it.kb; kbase < it.ke; kbase += kKeys, ++g) {
        const int st = g % kKStages;
        const int next_phys = (kbase + kKeys < it.ke) ? block_of(bt, nblk, kbase + kKeys) : 0;
        if (!__all_sync(0xffffffffu, mbar_wait(&bars->k_empty[st], ((g / kKStages) & 1) ^ 1, p.err))) {
          ok = false;
          break;
        }
        if (lane == 0) mbar_arrive_expect_tx(&bars->k_full[st], kTileBytes);
        __syncwarp();
        if (lane < nb) {
          uint8_t* d = smem + kKOff + st * kTileBytes + lane * p.bs * 128;
          tma_load_4d(d, &kmap, &bars->k_full[st], 0, it.kvh, 0, phys);
          tma_load_4d(d + kHalfKV, &kmap, &bars->k_full[st], 64, it.kvh, 0, phys);
        }
        phys = next_phys;
      }
    }
  } else if (warp == 11) {
    // ================================================================ V
    if (lane == 0) prefetch_tensormap(&vmap);
    int g = 0;
    bool ok = true;
    for (int c = 0; ok; ++c) {
      const int qb = c & 1;
      if (!__all_sync(0xffffffffu, mbar_wait(&bars->slot_full[qb], (c >> 1) & 1, p.err))) break;
      const bool done = slots[qb].done != 0;
      const WorkItem it = slots[qb].it;
      const int L = slots[qb].L;
      int phys = slots[qb].phys0[lane];
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->slot_free[qb]);
      if (done) break;
      const int nblk = (L + p.bs - 1) / p.bs;
      const int32_t* bt = p.block_tables + (int64_t)it.seq * p.max_blocks;
      for (int kbase = it.kb; kbase < it.ke; kbase += kKeys, ++g) {
        const int st = g % kVStages;
        const int next_phys = (kbase + kKeys < it.ke) ? block_of(bt, nblk, kbase + kKeys) : 0;
        // V stage g % 2 is free once P.V(g-2) is complete (phase of pv_done[g % 2])
        if (!__all_sync(0xffffffffu, mbar_wait(&bars->pv_done[st], ((g / kVStages) & 1) ^ 1, p.err))) {
          ok = false;
          break;
        }
        if (lane == 0) mbar_arrive_expect_tx(&bars->v_full[st], kTileBytes);
        __syncwarp();
        if (lane < nb) {
          uint8_t* d = smem + kVOff + st * kTileBytes + lane * p.bs * 128;
          tma_load_4d(d, &vmap, &bars->v_full[st], 0, it.kvh, 0, phys);
          tma_load_4d(d + kHalfKV, &vmap, &bars->v_full[st], 64, it.kvh, 0, phys);
        }
        phys = next_phys;
      }
    }
  } else if (warp == 1) {
    // ================================================================ Q K^T issuer
    if (lane == 0) {
      const uint64_t dq = desc_k(smem_base + kQOff);
      const uint64_t dk0 = desc_k(smem_base + kKOff);
      int gs = 0, s_item = -1, s_j = 0, s_nt = 0;
      for (;;) {
        if (s_j == s_nt) {  // next item: its Q tile loaded (its slot written before)
          ++s_item;
          const int qb = s_item & 1;
          if (!mbar_wait(&bars->q_full[qb], (s_item >> 1) & 1, p.err)) break;
          const bool done = slots[qb].done != 0;
          const int nt = (slots[qb].it.ke - slots[qb].it.kb + kKeys - 1) / kKeys;
          mbar_arrive(&bars->slot_free[qb]);
          if (done) break;
          s_nt = nt;
          s_j = 0;
        }
        const int sb = gs & 1, st = gs % kKStages;
        // S buffer sb: the softmax warps have read S(gs-2) from it; K(gs) loaded
        if (!mbar_test_wait3(&bars->s_free[sb], ((gs >> 1) & 1) ^ 1, &bars->k_full[st], (gs / kKStages) & 1,
                             &bars->k_full[st], (gs / kKStages) & 1) &&
            (!mbar_wait(&bars->s_free[sb], ((gs >> 1) & 1) ^ 1, p.err) ||
             !mbar_wait(&bars->k_full[st], (gs / kKStages) & 1, p.err)))
          break;
        tc_fence_after();
        const uint64_t dqb = desc_add(dq, (s_item & 1) * kQBytes);
        const uint64_t dk = desc_add(dk0, st * kTileBytes);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          umma_bf16(tmem + kSCol + 128 * sb, desc_add(dqb, (kk >> 2) * kHalf + (kk & 3) * 32),
                    desc_add(dk, (kk >> 2) * kHalfKV + (kk & 3) * 32), kIdescS, kk > 0 ? 1u : 0u);
        umma_commit(&bars->s_full[sb]);
        umma_commit(&bars->k_empty[st]);
        if (s_j == s_nt - 1) umma_commit(&bars->q_empty[s_item & 1]);  // Q no longer read by this item
        ++s_j;
        ++gs;
      }
    }
    __syncwarp();
  } else if (warp == 0) {
    // ================================================================ P.V issuer
    if (lane == 0) {
      const uint64_t dv0 = desc_v(smem_base + kVOff);
      int gp = 0;
      bool ok = true;
      for (int c = 0; ok; ++c) {
        const int qb = c & 1;
        if (!mbar_wait(&bars->slot_full[qb], (c >> 1) & 1, p.err)) break;
        const bool done = slots[qb].done != 0;
        const int nt = (slots[qb].it.ke - slots[qb].it.kb + kKeys - 1) / kKeys;
        mbar_arrive(&bars->slot_free[qb]);
        if (done) break;
        // O is about to be overwritten: item c-1's epilogue must have read it
        if (!mbar_wait(&bars->o_empty, (c & 1) ^ 1, p.err)) break;
        for (int j = 0; j < nt; ++j, ++gp) {
          const int pb = gp & 1, vst = gp % kVStages;
          // P(gp) written, V(gp) loaded
          if (!mbar_test_wait3(&bars->p_full[pb], (gp >> 1) & 1, &bars->v_full[vst], (gp / kVStages) & 1,
                               &bars->v_full[vst], (gp / kVStages) & 1) &&
              (!mbar_wait(&bars->p_full[pb], (gp >> 1) & 1, p.err) ||
               !mbar_wait(&bars->v_full[vst], (gp / kVStages) & 1, p.err))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t dv = desc_add(dv0, vst * kTileBytes);
#pragma unroll
          for (int kk = 0; kk < kKeys / 16; ++kk)
            umma_bf16_ts(tmem + kOCol, tmem + kPCol + 64 * pb + kk * 8, desc_add(dv, kk * 2048), kIdescO,
                         (j == 0 && kk == 0) ? 0u : 1u);
          umma_commit(&bars->pv_done[pb]);  // P.V(gp) complete: frees P buffer and V stage gp % 2
        }
      }
    }
    __syncwarp();
  } else {
    // ================================================================ softmax / epilogue
    const int q4 = warp & 3;
    const int h = (warp - 2) >> 2;  // key half of a tile (columns 64h .. 64h+63); output half 64h .. 64h+63
    const int r = q4 * 32 + lane;   // row of the tile == TMEM lane
    const int pair_bar = 1 + q4;    // warps (w, w+4) of one row quarter
    const uint32_t lane_base = tmem + ((uint32_t)(q4 * 32) << 16);
    float* red = reinterpret_cast<float*>(smem + kRedOff);
    int g = 0;
    bool ok = true;
    for (int c = 0; ok; ++c) {
      const int qb = c & 1;
      if (!__all_sync(0xffffffffu, mbar_wait(&bars->slot_full[qb], (c >> 1) & 1, p.err))) break;
      const ItemSlot& sl = slots[qb];
      const bool done = sl.done != 0;
      const WorkItem it = sl.it;
      const int L = sl.L, qstart = sl.qstart, n = sl.n;
      mbar_arrive(&bars->slot_free[qb]);
      if (done) break;
      const bool valid = r < it.nrows;
      const int row = it.row0 + r;
      const int tok = row / p.G, gh = row - tok * p.G;
      const int vis = valid ? min(it.ke, p.causal ? L - n + tok + 1 : L) : 0;
      float m_ref = -CUDART_INF_F, l = 0.f;
      const int ntiles = (it.ke - it.kb + kKeys - 1) / kKeys;
      for (int j = 0; j < ntiles; ++j, ++g) {
        const int sb = g & 1, vs = g % kVStages;
        const int kt = it.kb + j * kKeys;  // first key of the tile
        if (!__all_sync(0xffffffffu, mbar_wait(&bars->s_full[sb], (g >> 1) & 1, p.err))) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t sraw[64];
        tmem_ld32(lane_base + kSCol + 128 * sb + 64 * h, sraw);
        tmem_ld32(lane_base + kSCol + 128 * sb + 64 * h + 32, sraw + 32);
        tmem_wait_ld();
        tc_fence_before();
        mbar_arrive(&bars->s_free[sb]);  // S buffer sb may take S(g+2)
        const int nvis = vis - (kt + 64 * h);  // keys c < nvis of this half are visible
        if (nvis < 64) {
#pragma unroll
          for (int cc = 0; cc < 64; ++cc)
            if (cc >= nvis) sraw[cc] = __float_as_uint(-CUDART_INF_F);
        }
        float m4[4] = {-CUDART_INF_F, -CUDART_INF_F, -CUDART_INF_F, -CUDART_INF_F};
#pragma unroll
        for (int cc = 0; cc < 64; ++cc) m4[cc & 3] = fmaxf(m4[cc & 3], __uint_as_float(sraw[cc]));
        const float mloc = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));  // this half's max (raw S)
        float* redm = red + sb * 256;
        redm[h * 128 + r] = mloc;
        // P of keys 64h .. 64h+63: 2^(S scale_log2 - m) packed to bf16 pairs
        // (TMEM columns 32h .. 32h+31 of P buffer sb), ps2 their sums
        const f32x2 sc2 = pk2(p.scale_log2, p.scale_log2);
        uint32_t pk[32];
        f32x2 ps2[2];
        auto exps = [&](float m) {
          const float nm = m == -CUDART_INF_F ? 0.f : -m;
          const f32x2 nm2 = pk2(nm, nm);
          ps2[0] = ps2[1] = pk2(0.f, 0.f);
#pragma unroll
          for (int cc = 0; cc < 32; ++cc) {
            const float2 x = up2(fma2(pk2(__uint_as_float(sraw[2 * cc]), __uint_as_float(sraw[2 * cc + 1])), sc2, nm2));
            const float e0 = fast_exp2(x.x), e1 = fast_exp2(x.y);
            ps2[cc & 1] = add2(ps2[cc & 1], pk2(e0, e1));
            pk[cc] = pack_bf16(e0, e1);
          }
        };
        float alpha = 1.f;
        bool rescale = false;
        if (j == 0) {
          // first tile of the item: the row max first, then the exponentials
          named_barrier(pair_bar, 64);
          const float mx = fmaxf(mloc, redm[(h ^ 1) * 128 + r]) * p.scale_log2;
          if (mx > m_ref + kRescaleThreshold) {  // false while both are -inf
            alpha = fast_exp2(m_ref - mx);       // 0: m_ref is -inf here
            m_ref = mx;
          }
          exps(m_ref);
        } else {
          // The reference max of the earlier tiles is known, so the
          // exponentials go ahead of the pair's max exchange; they are redone
          // in the rare case that the row max exceeds the reference by more
          // than the threshold (or the row had no visible key before).
          exps(m_ref);
          named_barrier(pair_bar, 64);
          const float mx = fmaxf(mloc, redm[(h ^ 1) * 128 + r]) * p.scale_log2;
          if (mx > m_ref + kRescaleThreshold) {
            alpha = fast_exp2(m_ref - mx);  // 0 when m_ref is -inf
            rescale = m_ref != -CUDART_INF_F;
            m_ref = mx;
            exps(m_ref);
          }
        }
        // P buffer sb is free once the P.V of tile g-2, which read it, is done
        if (!__all_sync(0xffffffffu, mbar_wait(&bars->pv_done[sb], ((g >> 1) & 1) ^ 1, p.err))) {
          ok = false;
          break;
        }
        tmem_st32(lane_base + kPCol + 64 * sb + 32 * h, pk);
        {
          const float2 a = up2(ps2[0]), b = up2(ps2[1]);
          l = fmaf(l, alpha, (a.x + a.y) + (b.x + b.y));
        }
        if (__any_sync(0xffffffffu, rescale)) {
          // O must hold every earlier tile's P.V before it is scaled; the TMEM
          // accesses are warp-wide, rows that keep their max scale by 1
          // P.V(g-1) complete
          if (!__all_sync(0xffffffffu, mbar_wait(&bars->pv_done[sb ^ 1], ((g - 1) >> 1) & 1, p.err))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const float f = rescale ? alpha : 1.f;
#pragma unroll
          for (int cc = 0; cc < 2; ++cc) {
            uint32_t o[32];
            tmem_ld32(lane_base + kOCol + 64 * h + cc * 32, o);
            tmem_wait_ld();
#pragma unroll
            for (int t = 0; t < 32; ++t) o[t] = __float_as_uint(__uint_as_float(o[t]) * f);
            tmem_st32(lane_base + kOCol + 64 * h + cc * 32, o);
          }
        }
        if (kt + kKeys > L) {
          // keys at or past the sequence's end hold arbitrary bits: zero their V
          // rows (thread: key r of the tile, d-half h) so that 0 * V stays 0
          if (!__all_sync(0xffffffffu, mbar_wait(&bars->v_full[vs], (g / kVStages) & 1, p.err))) {
            ok = false;
            break;
          }
          if (kt + r >= L) {
            uint4* v0 = reinterpret_cast<uint4*>(smem + kVOff + vs * kTileBytes + h * kHalfKV + r * 128);
#pragma unroll
            for (int t = 0; t < 8; ++t) v0[t] = make_uint4(0, 0, 0, 0);
            fence_proxy_async_smem();
          }
        }
        tmem_wait_st();  // P (and a rescaled O) written
        tc_fence_before();
        mbar_arrive(&bars->p_full[sb]);
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
      // P.V of the item's last tile (g-1) complete
      if (!__all_sync(0xffffffffu, mbar_wait(&bars->pv_done[(g - 1) & 1], ((g - 1) >> 1) & 1, p.err))) break;
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
          uint32_t w[32];
#pragma unroll
          for (int u = 0; u < 32; ++u)
            w[u] = pack_bf16(__uint_as_float(o[2 * u]) * inv, __uint_as_float(o[2 * u + 1]) * inv);
          store_row128(orow, w, p.out_al32);
        } else {
          // this split's partial row: 256 bytes of fp32 (the workspace is 256-byte aligned)
          float* dst = p.part_acc + (int64_t)(it.part + r) * 128 + 64 * h;
#pragma unroll
          for (int u = 0; u < 8; ++u) st_global_v8(dst + 8 * u, o + 8 * u);
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
            for (int cc = 0; cc < 64; ++cc) acc[cc] = 0.f;
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
            uint32_t w[32];
#pragma unroll
            for (int u = 0; u < 32; ++u) w[u] = pack_bf16(acc[2 * u] * inv, acc[2 * u + 1] * inv);
            store_row128(orow, w, p.out_al32);
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
