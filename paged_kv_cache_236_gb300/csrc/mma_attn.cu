// Tensor-core paged attention for multi-token queries (prefill chunks,
// speculative verification): tcgen05.mma with TMEM accumulators.
//
// What it computes is the same as the other attention kernels ("Paged
// Attention 基础", section 2, steps 1-5; causal mask at each query's absolute
// position L - n + i; "ADR 004" Consequences: prefill and decode share one
// call), for a work item of up to 128 rows (query token, head-in-group) of one
// sequence and one kv head over keys [kb, ke):
//   S = Q K^T (128 rows x 128 keys per tile, fp32 in TMEM), online softmax in
//   registers, P (bf16) written to TMEM in 8-column pieces as the
//   exponentials produce them (the stores overlap the arithmetic, and a
//   thread holds 8 packed words instead of 32), O += P V (fp32 in TMEM; the tensor
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
// Roles (512 threads, one CTA per SM, persistent; items are taken from an
// atomic counter in the planner's largest-first order, so SMs that run
// slower take fewer):
//   warp 0     the thread issuing P.V (O += P V, P from TMEM, V from shared memory);
//   warp 1     TMEM allocation and the thread issuing Q K^T (S = Q K^T);
//   warps 2-3  K producers, one per 64-column half: per tile one
//              {64, 1, block_size, 1} box of the pool [NB, bs, Hkv, D] per
//              physical block (128-byte swizzle, the layout the tensor core
//              reads), block ids loaded a tile ahead;
//   warps 4-11 softmax / correction / epilogue: two threads per row (TMEM
//              lane), warps 4-7 on key columns 0-63 of a tile, warps 8-11 on
//              64-127; a pair exchanges row maxima (and at the end row sums)
//              through shared memory;
//   warps 12-13 V producers, the same boxes from the V pool;
//   warp 14    item fetch, Q and output stores: publishes each item in a
//              slot of shared memory (with the block ids of its first key
//              tile), then loads its Q tile (3-D box {64, G heads, 128/G
//              tokens} of q [T, Hq, D], two 64-column halves).  Before a Q
//              tile buffer takes a new item it stores, with two TMA stores of
//              the same boxes of out, the output tile that the epilogue of
//              the buffer's previous item left there: a finished 128-row tile
//              (whole tokens x G heads) is 32 KB that per-row stores would
//              write as 32-byte pieces 256 bytes to 8 KB apart.
// One warp's tensor copies of these 2 KB boxes are processed at about one
// box per 100 cycles whatever the number of issuing lanes, and copies
// completing on one barrier add up slower than on separate ones, so each
// 64-column half of K and of V has its own producer warp and barrier: four
// warps together supply the 64 KB of K and V a tile needs at the tensor
// core's pace.
// Shared memory: 2 Q tiles (64 KB), a 3-stage ring of K tiles (96 KB) and a
// 2-stage ring of V tiles (64 KB); K of a tile is released when its Q K^T is
// done, V when its P.V is done (K is needed two tiles ahead of V).
// TMEM (512 columns): S double-buffered in [0,256), P (32 columns of packed
// bf16 per 64 keys) double-buffered in [256,384), O in [384,512).
//
// The running max used for the exponentials is only raised when a tile's row
// maximum exceeds it by more than 8 (log2 units), so O is rescaled in TMEM
// rarely; P stays <= 2^8 and the result is exact up to rounding.
//
// Beside the decode kernel: every CTA signals its dependent (the decode
// kernel of the same call) as soon as it has seen the plan, and CTAs at or
// past the plan's mma_ctas take no items, so that the decode kernel's CTAs
// take their SMs and both kernels run at once on disjoint SMs.
//
// Shared-prefix items: an item whose rows are those of a run of sequences
// sharing leading blocks (their tokens are contiguous in q, from the run's
// first sequence) over keys of that prefix.  It writes partial rows and no
// merge; the decode kernel folds them into each member's rows.
//
// Bounded waits: every mbarrier wait gives up after the launch's limit
// (default 2 s), sets PKV_DEVERR_TIMEOUT and makes its role leave; a role
// that leaves first waits (bounded) for the copies or MMAs it has in flight,
// so that TMEM and shared memory are not released under them.  The roles
// that wait on one that left run out in turn, in parallel (no CTA-wide abort
// flag: reading one inside the waits cost 8 % of the prefill rate on GB300).  The softmax warps
// settle failures among themselves (see there); no warp is left at a named
// barrier waiting for one that left.  The kernel instance with kFaultHook
// (used only when a test sets the fault hook) skips one K copy so that the
// waits for it run out.
#include <math_constants.h>

#include "pkv_device.cuh"
#include "pkv_internal.h"
#include "pkv_tc.cuh"

namespace pkv {
namespace {

constexpr int kThreads = 512;
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
constexpr int kNumBars = 8 + 3 * kKStages + 2 * kVStages + 8 + 1 + 2;
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
// Register split between warpgroups (setmaxnreg): warpgroups 0 and 3 (MMA
// issuers, producers, item fetch) give up registers that warpgroups 1 and 2
// (softmax) take.  The sum must stay within what the block is launched with
// (kThreads x the kernel's register count); the launcher checks the count.
constexpr int kRegsLight = 64, kRegsSoftmax = 184;
static_assert(2 * 128 * (kRegsLight + kRegsSoftmax) <= kThreads * 128, "register split above 128 per thread");

constexpr uint32_t kIdescS = idesc_bf16(128, kKeys, false, false);
// P.V with N = head_dim (64 or 128)
template <int D>
constexpr uint32_t kIdescO = idesc_bf16(128, D, false, true);

// V as the B of P.V (MN-major): the two 64-column halves are kHalfKV apart,
// 8-key groups 1024 bytes apart.
__device__ __forceinline__ uint64_t desc_v(uint32_t saddr) { return smem_desc(saddr, kHalfKV, 1024); }

struct Bars {
  uint64_t q_full[2], q_empty[2], slot_full[2], slot_free[2];
  uint64_t k_full[kKStages][2], k_empty[kKStages];  // k_full[stage][64-column half]
  uint64_t v_full[kVStages][2];
  // s_full[b], phase n: S of tile 2n+b complete; s_free[b]: the softmax
  // warps have read it.  pv_done[b], phase n: the P.V of tile 2n+b complete,
  // and with it every earlier P.V.
  uint64_t s_full[2], s_free[2], pv_done[2], p_full[2];
  uint64_t o_empty;
  // o_staged[b], phase n: the epilogue of item 2n+b has left its output tile
  // in Q buffer b (or written it directly)
  uint64_t o_staged[2];
};

// An item's description, published by the item-fetching warp before its Q
// tile is loaded (slot_full), with the block ids of its first key tile.
struct alignas(16) ItemSlot {
  WorkItem it;
  int L, qstart, n, done;
  int phys0[32];
};
// readers of a slot: the 256 softmax threads, the two MMA-issuing threads, the four K / V producers
constexpr int kSlotReaders = 256 + 1 + 1 + 4;

static_assert(sizeof(ItemSlot) == 176, "item slot");
static_assert(sizeof(Bars) == kNumBars * 8, "barrier block");
static_assert(kVStages == 2, "V stage t % 2 is released by the P.V barrier of tile t");
static_assert(kSmem <= 232448, "shared memory");
static_assert(kKOff % 1024 == 0 && kVOff % 1024 == 0 && kTileBytes % 1024 == 0 && kQBytes % 1024 == 0,
              "swizzled tiles");
static_assert(kBarOff % 8 == 0 && kSlotOff % alignof(ItemSlot) == 0 && kRedOff % 16 == 0, "alignment");

// N bf16 (2N bytes) of an output row, packed in pairs in w: 32-byte stores
// when the output is 32-byte aligned, else 16-byte ones.
template <int N>
__device__ __forceinline__ void store_row(__nv_bfloat16* dst, const uint32_t* w, int al32) {
  if (al32) {
#pragma unroll
    for (int u = 0; u < N / 16; ++u) st_global_v8(dst + 16 * u, w + 8 * u);
  } else {
#pragma unroll
    for (int u = 0; u < N / 8; ++u)
      *reinterpret_cast<uint4*>(dst + 8 * u) = make_uint4(w[4 * u], w[4 * u + 1], w[4 * u + 2], w[4 * u + 3]);
  }
}

// D: head_dim, 64 or 128 (one or two 64-column halves of Q, K, V and the
// output; the shared-memory and TMEM layouts are those of 128, with the
// second halves unused at 64).  Each softmax thread owns D / 2 output
// columns of its row.
template <int D, bool kFaultHook>
__global__ void __launch_bounds__(kThreads, 1) mma_attn_kernel(const AttnParams p,
                                                               const __grid_constant__ CUtensorMap qmap,
                                                               const __grid_constant__ CUtensorMap kmap,
                                                               const __grid_constant__ CUtensorMap vmap,
                                                               const __grid_constant__ CUtensorMap omap) {
  constexpr int kNH = D / 64;   // 64-column halves
  constexpr int kOC = D / 2;    // output columns per softmax thread
  extern __shared__ __align__(1024) uint8_t smem[];
  if (smem_u32(smem) & 1023u) {  // uniform: every thread returns before any barrier
    if (threadIdx.x == 0) raise_error(p.err, PKV_DEVERR_INTERNAL);
    return;
  }
  Bars* bars = reinterpret_cast<Bars*>(smem + kBarOff);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kBarOff + kNumBars * 8);
  ItemSlot* slots = reinterpret_cast<ItemSlot*>(smem + kSlotOff);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const WaitCtl wc{p.err, wait_limit(p.wait_ns)};

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
      mbar_init(&bars->k_full[s][0], 1);
      mbar_init(&bars->k_full[s][1], 1);
      mbar_init(&bars->k_empty[s], 1);
    }
    for (int s = 0; s < kVStages; ++s) {
      mbar_init(&bars->v_full[s][0], 1);
      mbar_init(&bars->v_full[s][1], 1);
    }
    mbar_init(&bars->o_empty, 256);
    mbar_init(&bars->o_staged[0], 256);
    mbar_init(&bars->o_staged[1], 256);
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
  // CTAs past the plan's mma_ctas leave their SMs to the decode kernel, which
  // may start once every CTA here has seen the plan (signalled just below)
  const bool active = blockIdx.x < p.header->mma_ctas;
  pdl_launch_dependents();
  const uint32_t tmem = *tmem_slot;
  const uint32_t smem_base = smem_u32(smem);

  // One counter g numbers the key tiles this CTA processes (across items): K
  // stage g % 3 (parity (g / 3) & 1), V stage g % 2 (parity (g / 2) & 1), S
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

  // The branches below are per warpgroup first (the register split is a
  // warpgroup-wide instruction), then per warp.
  if (!active) {
    // nothing: straight to the teardown
  } else if (warp < 4 || warp >= 12) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsLight));
    if (warp == 14) {
      // ================================================================ item fetch, Q, output stores
      if (lane == 0) {
        prefetch_tensormap(&qmap);
        prefetch_tensormap(&omap);
      }
      // where the output tile staged in Q buffer b goes: token and head
      // coordinates of its TMA stores, token -1 when the epilogue wrote it itself
      int otok0 = -1, otok1 = -1, ohead0 = 0, ohead1 = 0;
      auto store_staged = [&](int ci) -> bool {  // item ci's output, once its epilogue is done
        const int b = ci & 1;
        if (!__all_sync(0xffffffffu, mbar_wait(&bars->o_staged[b], (ci >> 1) & 1, wc))) return false;
        const int tok = b ? otok1 : otok0, head = b ? ohead1 : ohead0;
        if (lane == 0 && tok >= 0) {
          tma_store_3d(&omap, smem + kQOff + b * kQBytes, 0, head, tok);
          if constexpr (kNH == 2) tma_store_3d(&omap, smem + kQOff + b * kQBytes + kHalf, 64, head, tok);
          bulk_commit_group();
          bulk_wait_read_all();  // the buffer may take the next Q tile
        }
        __syncwarp();
        return true;
      };
      int c = 0, q_last = -1;  // the last item whose Q tile was loaded
      bool ok = true;
      for (;; ++c) {
        const int qb = c & 1;
        // Item c is taken from the queue once item c-2's last Q K^T is
        // complete (Q tile qb free) and every reader has taken item c-2's
        // description (slot qb free): while item c-2 ends, item c-1 waits
        // with its Q loaded.  Taking items no earlier keeps the queue's
        // largest-first order close to the order in which the SMs fall idle,
        // which is what keeps the tail short.
        if (!__all_sync(0xffffffffu, mbar_wait(&bars->q_empty[qb], ((c >> 1) & 1) ^ 1, wc) &&
                                         mbar_wait(&bars->slot_free[qb], ((c >> 1) & 1) ^ 1, wc))) {
          ok = false;
          break;
        }
        int idx = 0;
        if (lane == 0) idx = atomicAdd(p.counter, 1);
        idx = __shfl_sync(0xffffffffu, idx, 0);
        const bool done = idx >= n_items;
        ItemSlot& sl = slots[qb];
        WorkItem it{};
        int qstart = 0;
        if (done) {
          if (lane == 0) sl.done = 1;
        } else {
          it = p.items[idx];
          const int L = p.context_lens[it.seq];
          qstart = p.query_start_loc[it.seq];
          const int nblk = (L + p.bs - 1) / p.bs;
          const int32_t* bt = p.block_tables + (int64_t)it.seq * p.max_blocks;
          sl.phys0[lane] = block_of(bt, nblk, it.kb);
          if (lane == 0) {
            sl.it = it;
            sl.L = L;
            sl.qstart = qstart;
            sl.n = p.query_start_loc[it.seq + 1] - qstart;
            sl.done = 0;
          }
        }
        mbar_arrive(&bars->slot_full[qb]);  // every lane, after its own writes (count 32)
        // Q tile qb: item c-2's output, staged there by its epilogue, read out
        if (c >= 2 && !store_staged(c - 2)) {
          ok = false;
          break;
        }
        if (done) {
          if (lane == 0) mbar_arrive(&bars->q_full[qb]);
          break;
        }
        // a full tile of whole tokens, not a split: its epilogue stages the output
        const int tok = (it.nrows == p.mma_unit_rows && it.part < 0) ? qstart + it.row0 / p.G : -1;
        if (qb) {
          otok1 = tok;
          ohead1 = it.kvh * p.G;
        } else {
          otok0 = tok;
          ohead0 = it.kvh * p.G;
        }
        if (lane == 0) {
          // the Q box: {64, G, floor(128 / G)} (whole tokens, up to 128 rows)
          mbar_arrive_expect_tx(&bars->q_full[qb], kNH * 128 * (kMmaRows / p.G) * p.G);
          const int tok0 = qstart + it.row0 / p.G;
          tma_load_3d(smem + kQOff + qb * kQBytes, &qmap, &bars->q_full[qb], 0, it.kvh * p.G, tok0);
          if constexpr (kNH == 2)
            tma_load_3d(smem + kQOff + qb * kQBytes + kHalf, &qmap, &bars->q_full[qb], 64, it.kvh * p.G, tok0);
        }
        q_last = c;
      }
      if (ok && c >= 1) store_staged(c - 1);  // the last item's output
      // leaving early: the last Q tile's copy must have landed before the CTA exits
      if (!ok && q_last >= 0) __all_sync(0xffffffffu, mbar_wait(&bars->q_full[q_last & 1], (q_last >> 1) & 1, wc));
      if (lane == 0) bulk_wait_all();
    } else if (warp == 2 || warp == 3 || warp == 12 || warp == 13) {
      // ================================================================ K / V producers
      const bool is_v = warp >= 12;
      const int hh = warp & 1;  // 64-column half
      const CUtensorMap* map = is_v ? &vmap : &kmap;
      if (lane == 0) prefetch_tensormap(map);
      const int nst = is_v ? kVStages : kKStages;
      uint8_t* const ring = smem + (is_v ? kVOff : kKOff) + hh * kHalfKV;
      int g = 0;
      bool ok = true;
      // leaving early: wait (bounded) until the copies of the tiles issued
      // last have landed
      auto drain = [&]() {
        for (int j = max(0, g - nst); j < g; ++j)
          __all_sync(0xffffffffu, mbar_wait(is_v ? &bars->v_full[j % nst][hh] : &bars->k_full[j % nst][hh],
                                            (j / nst) & 1, wc));
      };
      for (int c = 0; ok; ++c) {
        const int qb = c & 1;
        if (!__all_sync(0xffffffffu, mbar_wait(&bars->slot_full[qb], (c >> 1) & 1, wc))) {
          ok = false;
          break;
        }
        const bool done = slots[qb].done != 0;
        const WorkItem it = slots[qb].it;
        const int L = slots[qb].L;
        int phys = slots[qb].phys0[lane];
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->slot_free[qb]);
        if (done) break;
        if (hh >= kNH) continue;  // head_dim 64: the second half does not exist
        const int nblk = (L + p.bs - 1) / p.bs;
        const int32_t* bt = p.block_tables + (int64_t)it.seq * p.max_blocks;
        for (int kbase = it.kb; kbase < it.ke; kbase += kKeys, ++g) {
          const int st = g % nst, ph = (g / nst) & 1;
          const int next_phys = (kbase + kKeys < it.ke) ? block_of(bt, nblk, kbase + kKeys) : 0;
          // K stage g % 3 is free once Q K^T(g-3) is complete; V stage g % 2
          // once P.V(g-2) is complete (phase of pv_done[g % 2])
          if (!__all_sync(0xffffffffu, mbar_wait(is_v ? &bars->pv_done[st] : &bars->k_empty[st], ph ^ 1, wc))) {
            ok = false;
            break;
          }
          uint64_t* full = is_v ? &bars->v_full[st][hh] : &bars->k_full[st][hh];
          if (lane == 0) mbar_arrive_expect_tx(full, kHalfKV);
          __syncwarp();
          // testing only: one CTA's first K half of tile fault_tile - 1 is never
          // loaded, so the waits for it run out
          const bool skip = kFaultHook && p.fault_tile == g + 1 && !is_v && hh == 0 && blockIdx.x == 0;
          if (lane < nb && !skip) tma_load_4d(ring + st * kTileBytes + lane * p.bs * 128, map, full, 64 * hh, it.kvh, 0, phys);
          phys = next_phys;
        }
      }
      if (!ok) drain();
    } else if (warp == 1) {
      // ================================================================ Q K^T issuer
      if (lane == 0) {
        const uint64_t dq = desc_k(smem_base + kQOff);
        const uint64_t dk0 = desc_k(smem_base + kKOff);
        int gs = 0, s_item = -1, s_j = 0, s_nt = 0;
        bool ok = true;
        for (;;) {
          if (s_j == s_nt) {  // next item: its Q tile loaded (its slot written before)
            ++s_item;
            const int qb = s_item & 1;
            if (!mbar_wait(&bars->q_full[qb], (s_item >> 1) & 1, wc)) {
              ok = false;
              break;
            }
            const bool done = slots[qb].done != 0;
            const int nt = (slots[qb].it.ke - slots[qb].it.kb + kKeys - 1) / kKeys;
            mbar_arrive(&bars->slot_free[qb]);
            if (done) break;
            s_nt = nt;
            s_j = 0;
          }
          const int sb = gs & 1, st = gs % kKStages;
          // S buffer sb: the softmax warps have read S(gs-2) from it; both halves of K(gs) loaded
          const uint32_t kph = (gs / kKStages) & 1;
          uint64_t* const kf1 = &bars->k_full[st][kNH - 1];  // the second half's barrier (the first at head_dim 64)
          if (!mbar_test_wait3(&bars->s_free[sb], ((gs >> 1) & 1) ^ 1, &bars->k_full[st][0], kph, kf1, kph) &&
              (!mbar_wait(&bars->s_free[sb], ((gs >> 1) & 1) ^ 1, wc) ||
               !mbar_wait(&bars->k_full[st][0], kph, wc) || !mbar_wait(kf1, kph, wc))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t dqb = desc_add(dq, (s_item & 1) * kQBytes);
          const uint64_t dk = desc_add(dk0, st * kTileBytes);
  #pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            umma_bf16(tmem + kSCol + 128 * sb, desc_add(dqb, (kk >> 2) * kHalf + (kk & 3) * 32),
                      desc_add(dk, (kk >> 2) * kHalfKV + (kk & 3) * 32), kIdescS, kk > 0 ? 1u : 0u);
          umma_commit(&bars->s_full[sb]);
          umma_commit(&bars->k_empty[st]);
          if (s_j == s_nt - 1) umma_commit(&bars->q_empty[s_item & 1]);  // Q no longer read by this item
          ++s_j;
          ++gs;
        }
        // leaving early: the S MMAs already issued finish before TMEM is freed
        if (!ok && gs > 0) mbar_wait(&bars->s_full[(gs - 1) & 1], ((gs - 1) >> 1) & 1, wc);
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
          if (!mbar_wait(&bars->slot_full[qb], (c >> 1) & 1, wc)) {
            ok = false;
            break;
          }
          const bool done = slots[qb].done != 0;
          const int nt = (slots[qb].it.ke - slots[qb].it.kb + kKeys - 1) / kKeys;
          mbar_arrive(&bars->slot_free[qb]);
          if (done) break;
          // O is about to be overwritten: item c-1's epilogue must have read it
          if (!mbar_wait(&bars->o_empty, (c & 1) ^ 1, wc)) {
            ok = false;
            break;
          }
          for (int j = 0; j < nt; ++j, ++gp) {
            const int pb = gp & 1, vst = gp % kVStages;
            // P(gp) written, both halves of V(gp) loaded
            const uint32_t vph = (gp / kVStages) & 1;
            uint64_t* const vf1 = &bars->v_full[vst][kNH - 1];
            if (!mbar_test_wait3(&bars->p_full[pb], (gp >> 1) & 1, &bars->v_full[vst][0], vph, vf1, vph) &&
                (!mbar_wait(&bars->p_full[pb], (gp >> 1) & 1, wc) || !mbar_wait(&bars->v_full[vst][0], vph, wc) ||
                 !mbar_wait(vf1, vph, wc))) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint64_t dv = desc_add(dv0, vst * kTileBytes);
  #pragma unroll
            for (int kk = 0; kk < kKeys / 16; ++kk)
              umma_bf16_ts(tmem + kOCol, tmem + kPCol + 64 * pb + kk * 8, desc_add(dv, kk * 2048), kIdescO<D>,
                           (j == 0 && kk == 0) ? 0u : 1u);
            umma_commit(&bars->pv_done[pb]);  // P.V(gp) complete: frees P buffer and V stage gp % 2
          }
        }
        // leaving early: the P.V MMAs already issued finish before TMEM is freed
        if (!ok && gp > 0) mbar_wait(&bars->pv_done[(gp - 1) & 1], ((gp - 1) >> 1) & 1, wc);
      }
      __syncwarp();
    }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsSoftmax));
    // ================================================================ softmax / epilogue
    const int q4 = warp & 3;
    const int h = (warp - 4) >> 2;  // key half of a tile (columns 64h .. 64h+63); output half 64h .. 64h+63
    const int r = q4 * 32 + lane;   // row of the tile == TMEM lane
    const int pair_bar = 1 + q4;    // warps (w, w+4) of one row quarter
    const uint32_t lane_base = tmem + ((uint32_t)(q4 * 32) << 16);
    float* red = reinterpret_cast<float*>(smem + kRedOff);
    // A failed wait (warp-uniform) ends the warp's work on the item at once;
    // it then takes the pair barriers the item still owes its partner
    // (ntiles + 2 per item in all), so the partner never waits for a warp
    // that left: the partner finishes the item, or gives up in turn when a
    // wait of its own runs out.  All 8 warps then agree at an OR-reducing
    // barrier (id 6)
    // that each reaches once at the end of every item: there they all go on
    // to the stores, or all leave.
    int g = 0;
    for (int c = 0;; ++c) {
      const int qb = c & 1;
      if (barrier_any(6, 256, !__all_sync(0xffffffffu, mbar_wait(&bars->slot_full[qb], (c >> 1) & 1, wc)))) break;
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
      int owe = -1;  // after a failed wait: the pair barriers of the item not yet taken
      const int ntiles = (it.ke - it.kb + kKeys - 1) / kKeys;
      for (int j = 0; j < ntiles; ++j, ++g) {
        const int sb = g & 1, vs = g % kVStages;
        const int kt = it.kb + j * kKeys;  // first key of the tile
        if (!__all_sync(0xffffffffu, mbar_wait(&bars->s_full[sb], (g >> 1) & 1, wc))) {
          owe = ntiles - j + 2;
          break;
        }
        tc_fence_after();
        uint32_t sraw[64];
        tmem_ld32(lane_base + kSCol + 128 * sb + 64 * h, sraw);
        tmem_ld32(lane_base + kSCol + 128 * sb + 64 * h + 32, sraw + 32);
        tmem_wait_ld();
        tc_fence_before();
        mbar_arrive(&bars->s_free[sb]);  // S buffer sb may take S(g+2)
        // P buffer sb is free once the P.V of tile g-2, which read it, is done;
        // the exponentials below write P to it in 8-column pieces
        if (!__all_sync(0xffffffffu, mbar_wait(&bars->pv_done[sb], ((g >> 1) & 1) ^ 1, wc))) {
          owe = ntiles - j + 2;
          break;
        }
        const int nvis = vis - (kt + 64 * h);  // keys c < nvis of this half are visible
        if (nvis < 64) {
#pragma unroll
          for (int cc = 0; cc < 64; ++cc)
            if (cc >= nvis) sraw[cc] = __float_as_uint(-CUDART_INF_F);
        }
        // this half's max (raw S): four chains of three-operand max, two values a step
        float m4[4] = {-CUDART_INF_F, -CUDART_INF_F, -CUDART_INF_F, -CUDART_INF_F};
#pragma unroll
        for (int cc = 0; cc < 64; cc += 2)
          m4[(cc >> 1) & 3] =
              fmax3(m4[(cc >> 1) & 3], __uint_as_float(sraw[cc]), __uint_as_float(sraw[cc + 1]));
        const float mloc = fmaxf(fmax3(m4[0], m4[1], m4[2]), m4[3]);
        float* redm = red + sb * 256;
        redm[h * 128 + r] = mloc;
        // P of keys 64h .. 64h+63: 2^(S scale_log2 - m) packed to bf16 pairs
        // (TMEM columns 32h .. 32h+31 of P buffer sb), ps2 their sums
        const f32x2 sc2 = pk2(p.scale_log2, p.scale_log2);
        f32x2 ps2[2];
        auto exps = [&](float m) {
          const float nm = m == -CUDART_INF_F ? 0.f : -m;
          const f32x2 nm2 = pk2(nm, nm);
          ps2[0] = ps2[1] = pk2(0.f, 0.f);
#pragma unroll
          for (int grp = 0; grp < 4; ++grp) {
            uint32_t pk[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
              const int cc = grp * 8 + u;
              const float2 x = up2(fma2(pk2(__uint_as_float(sraw[2 * cc]), __uint_as_float(sraw[2 * cc + 1])), sc2, nm2));
              const float e0 = fast_exp2(x.x), e1 = fast_exp2(x.y);
              ps2[cc & 1] = add2(ps2[cc & 1], pk2(e0, e1));
              pk[u] = pack_bf16(e0, e1);
            }
            tmem_st8(lane_base + kPCol + 64 * sb + 32 * h + 8 * grp, pk);
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
            tmem_wait_st();  // the first pass's P pieces land before they are rewritten
            exps(m_ref);
          }
        }
        {
          const float2 a = up2(ps2[0]), b = up2(ps2[1]);
          l = fmaf(l, alpha, (a.x + a.y) + (b.x + b.y));
        }
        if (__any_sync(0xffffffffu, rescale)) {
          // O must hold every earlier tile's P.V before it is scaled; the TMEM
          // accesses are warp-wide, rows that keep their max scale by 1
          // P.V(g-1) complete
          if (!__all_sync(0xffffffffu, mbar_wait(&bars->pv_done[sb ^ 1], ((g - 1) >> 1) & 1, wc))) {
            owe = ntiles - j + 1;
            break;
          }
          tc_fence_after();
          const float f = rescale ? alpha : 1.f;
#pragma unroll
          for (int cc = 0; cc < kOC / 32; ++cc) {
            uint32_t o[32];
            tmem_ld32(lane_base + kOCol + kOC * h + cc * 32, o);
            tmem_wait_ld();
#pragma unroll
            for (int t = 0; t < 32; ++t) o[t] = __float_as_uint(__uint_as_float(o[t]) * f);
            tmem_st32(lane_base + kOCol + kOC * h + cc * 32, o);
          }
        }
        if (kt + kKeys > L && h < kNH) {
          // keys at or past the sequence's end hold arbitrary bits: zero their V
          // rows (thread: key r of the tile, d-half h) so that 0 * V stays 0
          if (!__all_sync(0xffffffffu, mbar_wait(&bars->v_full[vs][h], (g / kVStages) & 1, wc))) {
            owe = ntiles - j + 1;
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
      // ---- epilogue: row sum of the pair, O (this thread's D / 2 output columns) / l.
      // The sums go through the max buffer the last tile did not use; the
      // second pair barrier keeps the next tile from overwriting them early.
      float ltot = 0.f;
      if (owe < 0) {
        float* reds = red + (g & 1) * 256;
        reds[h * 128 + r] = l;
        named_barrier(pair_bar, 64);
        ltot = l + reds[(h ^ 1) * 128 + r];
        named_barrier(pair_bar, 64);
        // P.V of the item's last tile (g-1) complete
        if (!__all_sync(0xffffffffu, mbar_wait(&bars->pv_done[(g - 1) & 1], ((g - 1) >> 1) & 1, wc))) owe = 0;
      }
      for (int k = 0; k < owe; ++k) named_barrier(pair_bar, 64);
      if (barrier_any(6, 256, owe >= 0)) break;
      tc_fence_after();
      uint32_t o[kOC];
#pragma unroll
      for (int cc = 0; cc < kOC / 32; ++cc) tmem_ld32(lane_base + kOCol + kOC * h + 32 * cc, o + 32 * cc);
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive(&bars->o_empty);
      // a full tile of whole tokens leaves through TMA stores from Q buffer qb
      // (its Q K^T are complete), in the Q tile's layout: row r, 16-byte
      // chunk j at chunk j ^ (r & 7) of the row (128-byte swizzle); this
      // thread's columns kOC * h .. are chunks (kOC * h % 64) / 8 .. of half
      // kOC * h / 64
      const bool staged = it.nrows == p.mma_unit_rows && it.part < 0;
      if (valid) {
        if (it.part < 0) {
          const float inv = 1.f / ltot;
          uint32_t w[kOC / 2];
#pragma unroll
          for (int u = 0; u < kOC / 2; ++u)
            w[u] = pack_bf16(__uint_as_float(o[2 * u]) * inv, __uint_as_float(o[2 * u + 1]) * inv);
          if (staged) {
            uint8_t* srow = smem + kQOff + qb * kQBytes + (kOC * h / 64) * kHalf + r * 128;
#pragma unroll
            for (int jj = 0; jj < kOC / 8; ++jj) {
              const int j = ((kOC * h) % 64) / 8 + jj;
              *reinterpret_cast<uint4*>(srow + ((j ^ (r & 7)) << 4)) =
                  make_uint4(w[4 * jj], w[4 * jj + 1], w[4 * jj + 2], w[4 * jj + 3]);
            }
          } else {
            __nv_bfloat16* orow = reinterpret_cast<__nv_bfloat16*>(p.out) +
                                  ((int64_t)(qstart + tok) * p.Hq + (int64_t)it.kvh * p.G + gh) * D + kOC * h;
            store_row<kOC>(orow, w, p.out_al32);
          }
        } else {
          // this split's partial row: D fp32 (the workspace is 256-byte aligned)
          float* dst = p.part_acc + (int64_t)(it.part + r) * D + kOC * h;
#pragma unroll
          for (int u = 0; u < kOC / 8; ++u) st_global_v8(dst + 8 * u, o + 8 * u);
          if (h == 0) p.part_ml[it.part + r] = make_float2(m_ref, ltot);
        }
      }
      if (staged) fence_proxy_async_smem();  // the staged rows, for the TMA stores
      mbar_arrive(&bars->o_staged[qb]);
      if (it.grp >= 0) {
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
            float acc[kOC];
#pragma unroll
            for (int cc = 0; cc < kOC; ++cc) acc[cc] = 0.f;
            for (int sp = 0; sp < gr.nsplit; ++sp) {
              const int slot = gr.part_base + sp * gr.nrows + r;
              const float2 ml = __ldcg(&p.part_ml[slot]);
              const float wt = fast_exp2(ml.x - Mu);
              lsum = fmaf(wt, ml.y, lsum);
              const float4* src = reinterpret_cast<const float4*>(p.part_acc + (int64_t)slot * D + kOC * h);
#pragma unroll
              for (int u = 0; u < kOC / 4; ++u) {
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
                                  ((int64_t)(qstart + gtok) * p.Hq + (int64_t)gr.kvh * p.G + ggh) * D + kOC * h;
            uint32_t w[kOC / 2];
#pragma unroll
            for (int u = 0; u < kOC / 2; ++u) w[u] = pack_bf16(acc[2 * u] * inv, acc[2 * u + 1] * inv);
            store_row<kOC>(orow, w, p.out_al32);
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

template <int D, bool kFaultHook>
cudaError_t launch_mma_t(const AttnParams& p, const CUtensorMap& qmap, const CUtensorMap& kmap,
                         const CUtensorMap& vmap, const CUtensorMap& omap, int grid, cudaStream_t s) {
  static unsigned long long done_mask = 0;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!(__atomic_load_n(&done_mask, __ATOMIC_ACQUIRE) & (1ull << dev))) {
    // the register split needs the block launched with 128 registers per thread
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, mma_attn_kernel<D, kFaultHook>);
    if (e != cudaSuccess) return e;
    if (fa.numRegs != 128) return cudaErrorInvalidConfiguration;
    e = cudaFuncSetAttribute(mma_attn_kernel<D, kFaultHook>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e != cudaSuccess) return e;
    __atomic_fetch_or(&done_mask, 1ull << dev, __ATOMIC_RELEASE);
  }
  if (p.no_wait) {
    // beside the decode kernel (p.no_wait): a plain launch, which starts once
    // the planner's grid has completed; started early, before the plan, it
    // delayed the pair on the mixed batch
    mma_attn_kernel<D, kFaultHook><<<dim3(grid), dim3(kThreads), kSmem, s>>>(p, qmap, kmap, vmap, omap);
    e = cudaGetLastError();
  } else {
    e = launch_pdl(mma_attn_kernel<D, kFaultHook>, dim3(grid), dim3(kThreads), kSmem, s, p, qmap, kmap, vmap, omap);
  }
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace

cudaError_t launch_mma(const AttnParams& p, const CUtensorMap& qmap, const CUtensorMap& kmap, const CUtensorMap& vmap,
                       const CUtensorMap& omap, int grid, cudaStream_t s) {
  if (p.fault_tile)  // testing only
    return p.D == 64 ? launch_mma_t<64, true>(p, qmap, kmap, vmap, omap, grid, s)
                     : launch_mma_t<128, true>(p, qmap, kmap, vmap, omap, grid, s);
  return p.D == 64 ? launch_mma_t<64, false>(p, qmap, kmap, vmap, omap, grid, s)
                   : launch_mma_t<128, false>(p, qmap, kmap, vmap, omap, grid, s);
}

}  // namespace pkv
