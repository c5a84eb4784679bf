// Tensor-core paged attention for few rows per kv head (decode, short
// speculative windows): tcgen05.mma with the keys on the M axis.
//
// What it computes is the same as every other attention kernel here
// ("Paged Attention 基础", section 2, steps 1-5; causal mask at each query's
// absolute position L - n + i): for a work item of up to 16 rows (query
// token, head-in-group) of one sequence and one kv head over keys [kb, ke),
// softmax(scale * q k^T) v with a running (max, sum), normalised at the end,
// or a partial (m, l, acc) row for split-KV; the last split of a merge group
// to finish merges the group (atomic ticket, no waiting).
//
// Why tensor cores: decode reads every K/V byte once and does 4 FMAs per
// byte pair per query row; on CUDA cores the conversions, reductions and
// FMAs leave the SMs latency-bound below the HBM rate.  Here each 128-key
// tile costs two small MMAs, with the rows on N:
//   S^T [128 keys x 16 rows] = K [128 keys x 128 d] . Q^T        (A K-major, B K-major)
//   O^T [128 d x 16 rows]   += V^T [128 d x 128 keys] . P^T      (A MN-major, B K-major)
// so one thread per key does the softmax arithmetic for its key (16 values)
// and one thread per output column writes the result, coalesced.
//
// Roles (384 threads, one CTA per SM, persistent, items from an atomic
// counter in the planner's largest-first order):
//   warp 0    K producer: per 128-key tile one {64, 1, block_size, 1} box
//             per physical block and 64-column half of K (128-byte swizzle;
//             out-of-range boxes for blocks past the end read as zeros), and
//             an item's Q tile ({64, G, 16/G} box of q) with its first tile;
//             item descriptions travel in per-stage metadata;
//   warp 11   V producer, the same boxes of V.  One warp's tensor copies are
//             processed at about one 2 KB box per 100 cycles, under the
//             HBM rate an SM needs, so K and V are issued by two warps;
//   warp 1    TMEM allocation and the single thread issuing the MMAs; the
//             P.V of tile g goes as soon as its P is written, or after the
//             S of tile g+1 when K(g+1) lands first (a P.V held back behind
//             a late K would hold its K/V stage, and the ring runs dry);
//   warps 2-5 softmax (thread = key = TMEM lane);
//   warps 6-9 epilogue (thread = output column = TMEM lane of O^T);
//   warp 10   item fetch: shortly before the K producer needs the next item
//             (two tiles before the end of the current one), it takes it
//             from the queue and reads its record, its sequence's length and
//             query offset and the block ids of its first tile into a slot
//             in shared memory, so that the producers start an item's loads
//             without a chain of dependent global reads.
// Shared memory: 3 stages of K+V (192 KB), 2 Q tiles and 2 P tiles (4 KB
// each).  TMEM: S^T double-buffered in columns [0,32), O^T in [32,48).
//
// FP8 pools (E4M3 codes, one scale per pool), items of up to 8 rows: 512
// threads.  The producers load each tile's codes (one {128, 1, block_size,
// 1} box per block, 16 KB of K and 16 KB of V) into a 2-slot staging ring and
// run ahead of the MMAs; warps 12-15 convert a staged tile into the fp16 tile
// the MMAs read (E4M3 -> fp16 is exact, one instruction per two codes; the
// same 128-byte swizzle), and an item's Q tile from bf16 to fp16 in place.
// The MMAs then run on fp16 A and B; P is written as fp16.  Two fp16 stages,
// 4 Q tiles and 4 metadata slots (the producers are up to two tiles ahead).
// The K scale is in the logit scale, the V scale multiplies the output.
//
// Bounded waits (failure detection): every wait gives up after a time limit
// (2 s unless the call sets one); the roles that wait on one that gave up
// run out in turn, in parallel.  Waits whose outcome decides
// what a group of warps does next are settled across the group by a barrier
// that ORs the failures, so that all of the group's warps go on or all
// leave; nothing waits without a bound.  A producer that leaves first waits
// (bounded) for its copies in flight, and the MMA thread for its last MMAs;
// then every role meets at the end, where TMEM is freed.
//
// An unsplit item after a shared prefix (part < 0, merge group >= 0) folds
// the prefix's partial rows, written by the tensor-core kernel before this
// one ran, into its own rows in the epilogue; a split one leaves that to its
// group's merge, which folds in the splits and the prefix partials alike.
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <math_constants.h>

#include "pkv_device.cuh"
#include "pkv_internal.h"
#include "pkv_tc.cuh"

namespace pkv {
namespace {

constexpr int kMaxStages = 3;
constexpr int kKeys = kMmaTileKeys;            // 128 keys per tile
constexpr int kN = kTcDecRows;                 // 16 rows (MMA N)
constexpr int kTileBytes = kKeys * 128 * 2;    // one of K or V: 32 KB
constexpr int kStageBytes = 2 * kTileBytes;
constexpr int kCodeTile = kKeys * 128;         // one of K or V as E4M3 codes: 16 KB
constexpr int kQHalf = kN * 128;               // one 64-column half of the Q / P tiles (2 KB)
constexpr int kNumBars = 5 * kMaxStages + 2 * 8 + 4 + 2 + 1;
// The K producer asks for the next item when this many tiles of the current
// one are left to load: early enough to hide the fetch (a few dependent
// global reads), late enough that an SM does not hold an item for long
// while others fall idle at the end of the queue.
constexpr int kFetchLeadTiles = 2;

// Shared-memory layout.  bf16 pools: 3 stages of K+V.  FP8 pools: 2 stages
// of fp16 K+V (what the MMAs read) and 2 stages of staged codes (what TMA
// writes), and 4 more warps that convert the one into the other.
template <bool F8>
struct Lay {
  static constexpr int kThreads = F8 ? 512 : 384;
  static constexpr int kStages = F8 ? 2 : 3;
  // FP8: the producers run ahead of the fp16 stages on the staging ring, so
  // tile metadata and Q tiles live in 4 slots (a slot is rewritten only
  // after every reader of its previous tile is done with it)
  static constexpr int kMetaSlots = F8 ? 4 : kStages;
  static constexpr int kQBufs = F8 ? 4 : 2;
  static constexpr int kQOff = kStages * kStageBytes;
  static constexpr int kPOff = kQOff + kQBufs * 2 * kQHalf;
  static constexpr int kMetaOff = kPOff + 2 * 2 * kQHalf;
  static constexpr int kRedOff = kMetaOff + kMetaSlots * 64;
  static constexpr int kSlotOff = kRedOff + 2 * 4 * kN * 4;
  static constexpr int kISlotOff = kSlotOff + 2 * 256;  // 2 item slots
  static constexpr int kStgOff = (kISlotOff + 2 * 192 + 1023) & ~1023;
  static constexpr int kStgBytes = F8 ? kStages * 2 * kCodeTile : 0;
  static constexpr int kBarOff = F8 ? kStgOff + kStgBytes : kISlotOff + 2 * 192;
  static constexpr int kSmem = kBarOff + kNumBars * 8 + 16 + 1024;
};
static_assert(Lay<true>::kSmem <= 232448 && Lay<false>::kSmem <= 232448, "shared memory per CTA");
constexpr uint32_t kTmemCols = 64;
constexpr uint32_t kSCol = 0, kOCol = 32;
constexpr float kRescaleThreshold = 8.0f;  // log2 units
constexpr int kMetaDone = 2, kMetaLast = 1, kMetaFirst = 4;

constexpr uint32_t kIdescS = idesc_bf16(128, kN, false, false);
constexpr uint32_t kIdescO = idesc_bf16(128, kN, true, false);
// fp16 A and B (FP8 pools decode to fp16 exactly): the format fields are 0
constexpr uint32_t kIdescS16 = kIdescS & ~((7u << 7) | (7u << 10));
constexpr uint32_t kIdescO16 = kIdescO & ~((7u << 7) | (7u << 10));

struct alignas(16) Meta {
  int item, kbase, flags, seq;
  int kvh, row0, nrows, ke;
  int part, grp, L, n;
  int qstart, pad0, pad1, pad2;
};
static_assert(sizeof(Meta) == 64, "meta slot");

struct Bars {
  uint64_t k_full[kMaxStages], v_full[kMaxStages], kv_empty[kMaxStages];
  uint64_t kc_full[kMaxStages], vc_full[kMaxStages];  // FP8: fp16 K / V of the stage converted
  uint64_t s_full[2], s_free[2], p_full[2], pv_done[2];
  uint64_t o_full[2], o_empty[2], ml_full[2], ml_empty[2];
  uint64_t islot_full[2], islot_free[2];
  uint64_t stage_empty[2];  // FP8: a staging slot's codes converted (the producers may refill it)
  uint64_t fetch_go;        // phase c: the K producer is near the end of item c (fetch item c + 1)
};

// An item as the item-fetch warp hands it to the producer.
struct alignas(16) ItemSlot {
  WorkItem it;
  int idx, L, qstart, n;
  int done, pad[3];
  int phys0[32];  // physical block of each of the item's first tile's blocks
};
static_assert(sizeof(ItemSlot) == 192, "item slot");

// What the softmax warps hand the epilogue at an item's end.
struct alignas(16) EpSlot {
  Meta mt;
  float m[kN], l[kN];
  int done;
  int pad[15];
};
static_assert(sizeof(EpSlot) == 256, "epilogue slot");
static_assert(sizeof(Bars) == kNumBars * 8, "barrier block");

// A merge group as the planner wrote it, read from L2 (see no_wait).
__device__ __forceinline__ MergeGroup load_group(const MergeGroup* g) {
  static_assert(sizeof(MergeGroup) == 48, "merge group");
  const int4* src = reinterpret_cast<const int4*>(g);
  const int4 a = __ldcg(src), b = __ldcg(src + 1), c = __ldcg(src + 2);
  MergeGroup m;
  m.seq = a.x; m.kvh = a.y; m.row0 = a.z; m.nrows = a.w;
  m.nsplit = b.x; m.part_base = b.y; m.pre_base = b.z; m.pre_n = b.w;
  m.pre_stride = c.x; m.pad0 = c.y; m.pad1 = c.z; m.pad2 = c.w;
  return m;
}

// A warp waits for a phase; true for every lane only if it completed for all.
__device__ __forceinline__ bool wait_all(uint64_t* bar, uint32_t parity, const WaitCtl& w) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity, w));
}

// Reduce NR values per lane over the 32 lanes of a warp with `op`,
// transposing: the result returned by lane l is the reduction of value
// row_of(l) = l >> (5 - log2 NR), so NR values cost NR - 1 + 5 - log2 NR shuffles.
template <int NR, typename Op>
__device__ __forceinline__ float xreduce(float (&a)[NR], int lane, Op op) {
  constexpr int kLog = NR == 1 ? 0 : NR == 2 ? 1 : NR == 4 ? 2 : NR == 8 ? 3 : 4;
#pragma unroll
  for (int lvl = 0; lvl < kLog; ++lvl) {
    const int off = 16 >> lvl;
    const int half = NR >> (lvl + 1);
    const bool up = lane & off;
#pragma unroll
    for (int i = 0; i < half; ++i) {
      const float send = up ? a[i] : a[i + half];
      const float keep = up ? a[i + half] : a[i];
      a[i] = op(keep, __shfl_xor_sync(0xffffffffu, send, off));
    }
  }
  float x = a[0];
#pragma unroll
  for (int off = 16 >> kLog; off > 0; off >>= 1) x = op(x, __shfl_xor_sync(0xffffffffu, x, off));
  return x;
}

template <int NR>
__device__ __forceinline__ void tmem_ld_rows(uint32_t taddr, uint32_t (&v)[NR]) {
  if constexpr (NR == 4) tmem_ld4(taddr, v);
  else if constexpr (NR == 8) tmem_ld8(taddr, v);
  else tmem_ld16(taddr, v);
}
template <int NR>
__device__ __forceinline__ void tmem_st_rows(uint32_t taddr, const uint32_t (&v)[NR]) {
  if constexpr (NR == 4) tmem_st4(taddr, v);
  else if constexpr (NR == 8) tmem_st8(taddr, v);
  else tmem_st16(taddr, v);
}

struct MaxOp {
  __device__ __forceinline__ float operator()(float a, float b) const { return fmaxf(a, b); }
};
struct AddOp {
  __device__ __forceinline__ float operator()(float a, float b) const { return a + b; }
};

// Two E4M3 codes (low byte first) as an fp16 pair, exactly (every E4M3
// value is an fp16 value).
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two) {
  const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)two, __NV_E4M3);
  return (uint32_t)h.x | ((uint32_t)h.y << 16);
}

// One tile of codes (128 keys x 128 bytes, row-major) as the fp16 tile the
// MMAs read: two 64-column halves kHalf apart, key r's 16-byte chunk j at
// chunk j ^ (r & 7) of its 128-byte row (the 128-byte swizzle).  Thread c of
// the 128 converter threads takes 16-code chunks c, c + 128, ...
__device__ __forceinline__ void convert_tile(const uint8_t* src, uint8_t* dst, int c) {
#pragma unroll 2
  for (int u = c; u < kKeys * 8; u += 128) {
    const int key = u >> 3, ch = u & 7;
    const uint4 raw = *reinterpret_cast<const uint4*>(src + key * 128 + ch * 16);
    const uint32_t in[4] = {raw.x, raw.y, raw.z, raw.w};
    uint32_t w[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      w[2 * i] = e4m3x2_to_f16x2(in[i] & 0xFFFFu);
      w[2 * i + 1] = e4m3x2_to_f16x2(in[i] >> 16);
    }
    uint8_t* row = dst + (ch >> 2) * kHalf + key * 128;
    const int j0 = (ch & 3) * 2;
    *reinterpret_cast<uint4*>(row + ((j0 ^ (key & 7)) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
    *reinterpret_cast<uint4*>(row + (((j0 + 1) ^ (key & 7)) << 4)) = make_uint4(w[4], w[5], w[6], w[7]);
  }
}

// Eight bf16 values as eight fp16 values (round to nearest; magnitudes above
// 65504 become infinite).
__device__ __forceinline__ uint4 bf16x8_to_f16x8(uint4 v) {
  const uint32_t in[4] = {v.x, v.y, v.z, v.w};
  uint32_t out[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __half2 h = __floats2half2_rn(__uint_as_float(in[i] << 16), __uint_as_float(in[i] & 0xFFFF0000u));
    out[i] = *reinterpret_cast<const uint32_t*>(&h);
  }
  return make_uint4(out[0], out[1], out[2], out[3]);
}

// NR: rows per item (4, 8 or 16; the MMA's N stays 16, extra columns unused).
// F8: the pools hold E4M3 codes (q bf16): staged codes are converted to fp16
// tiles and the MMAs run on fp16 operands.
template <int NR, bool F8>
__global__ void __launch_bounds__(Lay<F8>::kThreads, 1) dectc_kernel(const AttnParams p,
                                                            const __grid_constant__ CUtensorMap qmap,
                                                            const __grid_constant__ CUtensorMap kmap,
                                                            const __grid_constant__ CUtensorMap vmap) {
  using Y = Lay<F8>;
  extern __shared__ __align__(16) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  Bars* bars = reinterpret_cast<Bars*>(smem + Y::kBarOff);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Y::kBarOff + kNumBars * 8);
  Meta* meta = reinterpret_cast<Meta*>(smem + Y::kMetaOff);
  float* red = reinterpret_cast<float*>(smem + Y::kRedOff);  // [2][4 warps][NR rows]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const WaitCtl wc{p.err, wait_limit(p.wait_ns)};

  if (threadIdx.x == 0) {
    for (int s = 0; s < Y::kStages; ++s) {
      mbar_init(&bars->k_full[s], 1);
      mbar_init(&bars->v_full[s], 1);
      mbar_init(&bars->kv_empty[s], 1);
      mbar_init(&bars->kc_full[s], 128);  // the 128 converter threads (FP8)
      mbar_init(&bars->vc_full[s], 128);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bars->s_full[b], 1);
      mbar_init(&bars->s_free[b], 128);
      mbar_init(&bars->p_full[b], 128);
      mbar_init(&bars->pv_done[b], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bars->o_full[b], 1);
      mbar_init(&bars->o_empty[b], 128);
      mbar_init(&bars->ml_full[b], 128);
      mbar_init(&bars->ml_empty[b], 128);
      mbar_init(&bars->islot_full[b], 32);
      mbar_init(&bars->islot_free[b], 2);  // both producers read the slot
      if (b == 0) mbar_init(&bars->fetch_go, 1);
      mbar_init(&bars->stage_empty[b], 128);
    }
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // The plan and the K/V write are complete and visible from here on: after
  // the wait for the preceding grid, or, beside the tensor-core kernel, from
  // launch (that kernel lets this one start only after seeing the plan); the
  // plan is then read from L2 (__ldcg), past any stale L1 line.
  if (!p.no_wait) pdl_wait();
  const int n_items = __ldcg(&p.header->n_dec);
  const uint32_t tmem = *tmem_slot;
  const uint32_t smem_base = smem_u32(smem);

  if (warp == 0 || warp == 11) {
    // ================================================================ K / V producers
    const bool vprod = warp == 11;
    if (lane == 0) {
      if (vprod) {
        prefetch_tensormap(&vmap);
      } else {
        prefetch_tensormap(&qmap);
        prefetch_tensormap(&kmap);
      }
    }
    const int nb_per_tile = kKeys / p.bs;
    const ItemSlot* islots = reinterpret_cast<const ItemSlot*>(smem + Y::kISlotOff);
    int g = 0;
    // On giving up: wait (bounded) until the copies of the tiles issued
    // last have landed, so that none is still in
    // flight into this CTA's shared memory when it exits.
    uint64_t* fullb = vprod ? bars->v_full : bars->k_full;
    auto drain = [&]() {
      for (int j = max(0, g - Y::kStages); j < g; ++j)
        __all_sync(0xffffffffu, mbar_wait(&fullb[j % Y::kStages], (j / Y::kStages) & 1, wc));
    };
    for (int it_cnt = 0;; ++it_cnt) {
      const int qb = it_cnt & 1;
      if (!wait_all(&bars->islot_full[qb], (it_cnt >> 1) & 1, wc)) {
        drain();
        break;
      }
      const ItemSlot& isl = islots[qb];
      const bool done = isl.done != 0;
      const WorkItem it = isl.it;
      const int idx = isl.idx, L = isl.L, qstart = isl.qstart, n = isl.n;
      int phys = isl.phys0[lane];
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->islot_free[qb]);
      if (done) {
        if (vprod) break;
        const int st = g % Y::kStages;
        if (!wait_all(F8 ? &bars->stage_empty[st] : &bars->kv_empty[st], ((g / Y::kStages) & 1) ^ 1, wc)) {
          drain();
          break;
        }
        const int mi = F8 ? (g & 3) : st;
        if (lane == 0) {
          meta[mi].item = -1;
          meta[mi].flags = kMetaDone;
          mbar_arrive(&bars->k_full[st]);
        }
        break;
      }
      const int nblk = (L + p.bs - 1) / p.bs;
      const int32_t* bt = p.block_tables + (int64_t)it.seq * p.max_blocks;
      auto block_of = [&](int kbase) -> int {  // physical block of this lane's block in the tile
        const int lb = kbase / p.bs + lane;
        int phys_ = (int)p.num_blocks;  // out of range: the box reads as zeros
        if (lane < nb_per_tile && lb < nblk) {
          const int b = __ldg(bt + lb);
          if (b >= 0 && (int64_t)b < p.num_blocks)
            phys_ = b;
          else
            raise_error(p.err, PKV_DEVERR_BLOCK_OUT_OF_RANGE);
        }
        return phys_;
      };
      bool ok = true;
      for (int kbase = it.kb; kbase < it.ke; kbase += kKeys, ++g) {
        const int st = g % Y::kStages;
        const bool first = kbase == it.kb;
        const int next_phys = (kbase + kKeys < it.ke) ? block_of(kbase + kKeys) : 0;
        // bf16: the stage's K/V tiles are free once its last P.V is done.
        // FP8: the staging slot is free once its codes are converted.
        if (!wait_all(F8 ? &bars->stage_empty[st] : &bars->kv_empty[st], ((g / Y::kStages) & 1) ^ 1, wc)) {
          ok = false;
          break;
        }
        if (!vprod && lane == 0 && it.ke - kbase <= kFetchLeadTiles * kKeys &&
            (first || it.ke - (kbase - kKeys) > kFetchLeadTiles * kKeys))
          mbar_arrive(&bars->fetch_go);  // once per item: the next one may be taken now
        if (!vprod && p.fault_tile == g + 1 && blockIdx.x == 0) {
          // testing only: this tile is never loaded, so the waits for it run out
          phys = next_phys;
          continue;
        }
        uint8_t* kd = smem + st * kStageBytes;
        uint8_t* vd = kd + kTileBytes;
        // FP8: the codes of K and V land in the staging area (one 128-byte
        // row per key, one box per block); the converter warps fill kd / vd
        uint8_t* kc8 = smem + Y::kStgOff + st * 2 * kCodeTile;
        uint8_t* vc8 = kc8 + kCodeTile;
        if (vprod) {
          if (lane == 0) mbar_arrive_expect_tx(&bars->v_full[st], F8 ? kCodeTile : kTileBytes);
          __syncwarp();
          if (lane < nb_per_tile) {
            const int row_off = lane * p.bs * 128;
            if constexpr (F8) {
              tma_load_4d(vc8 + row_off, &vmap, &bars->v_full[st], 0, it.kvh, 0, phys);
            } else {
              tma_load_4d(vd + row_off, &vmap, &bars->v_full[st], 0, it.kvh, 0, phys);
              tma_load_4d(vd + kHalf + row_off, &vmap, &bars->v_full[st], 64, it.kvh, 0, phys);
            }
          }
          phys = next_phys;
          continue;
        }
        if (lane == 0) {
          Meta& m = meta[F8 ? (g & 3) : st];
          m.item = idx;
          m.kbase = kbase;
          m.flags = ((kbase + kKeys >= it.ke) ? kMetaLast : 0) | (first ? kMetaFirst : 0);
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
          mbar_arrive_expect_tx(&bars->k_full[st], (F8 ? kCodeTile : kTileBytes) + (first ? 2 * kQHalf : 0));
          if (first) {
            // this item's Q rows: tokens row0/G .. of the item, G heads each
            uint8_t* qd = smem + Y::kQOff + (it_cnt & (Y::kQBufs - 1)) * 2 * kQHalf;
            const int tok0 = qstart + it.row0 / p.G;
            tma_load_3d(qd, &qmap, &bars->k_full[st], 0, it.kvh * p.G, tok0);
            tma_load_3d(qd + kQHalf, &qmap, &bars->k_full[st], 64, it.kvh * p.G, tok0);
          }
        }
        __syncwarp();
        if (lane < nb_per_tile) {
          const int row_off = lane * p.bs * 128;
          if constexpr (F8) {
            tma_load_4d(kc8 + row_off, &kmap, &bars->k_full[st], 0, it.kvh, 0, phys);
          } else {
            tma_load_4d(kd + row_off, &kmap, &bars->k_full[st], 0, it.kvh, 0, phys);
            tma_load_4d(kd + kHalf + row_off, &kmap, &bars->k_full[st], 64, it.kvh, 0, phys);
          }
        }
        phys = next_phys;
      }
      if (!ok) {
        drain();
        break;
      }
    }
  } else if (warp == 10) {
    // ================================================================ item fetch
    const int nb_per_tile = kKeys / p.bs;
    ItemSlot* islots = reinterpret_cast<ItemSlot*>(smem + Y::kISlotOff);
    for (int c = 0;; ++c) {
      const int qb = c & 1;
      // Item c is taken from the queue when the K producer is within
      // kFetchLeadTiles tiles of the end of item c-1, and once both
      // producers have taken item c-2 (freeing slot qb).  Taking items no
      // earlier keeps the queue's largest-first order close to the order in
      // which the SMs fall idle, so the SMs finish together.
      if (c >= 1 && !wait_all(&bars->fetch_go, (c - 1) & 1, wc)) break;
      if (c >= 2 && !wait_all(&bars->islot_free[(c - 2) & 1], ((c - 2) >> 1) & 1, wc)) break;
      int idx = 0;
      if (lane == 0) idx = atomicAdd(p.counter, 1);
      idx = __shfl_sync(0xffffffffu, idx, 0);
      ItemSlot& isl = islots[qb];
      if (idx >= n_items) {
        if (lane == 0) isl.done = 1;
        mbar_arrive(&bars->islot_full[qb]);  // every lane: count 32
        break;
      }
      WorkItem it;
      {
        const int4* src = reinterpret_cast<const int4*>(p.items + idx);
        const int4 a = __ldcg(src), b = __ldcg(src + 1);
        it.seq = a.x; it.kvh = a.y; it.row0 = a.z; it.nrows = a.w;
        it.kb = b.x; it.ke = b.y; it.part = b.z; it.grp = b.w;
      }
      const int L = p.context_lens[it.seq];
      const int qstart = p.query_start_loc[it.seq];
      const int n = p.query_start_loc[it.seq + 1] - qstart;
      const int nblk = (L + p.bs - 1) / p.bs;
      const int lb = it.kb / p.bs + lane;
      int phys = (int)p.num_blocks;  // out of range: the box reads as zeros
      if (lane < nb_per_tile && lb < nblk) {
        const int b = __ldg(p.block_tables + (int64_t)it.seq * p.max_blocks + lb);
        if (b >= 0 && (int64_t)b < p.num_blocks)
          phys = b;
        else
          raise_error(p.err, PKV_DEVERR_BLOCK_OUT_OF_RANGE);
      }
      isl.phys0[lane] = phys;
      if (lane == 0) {
        isl.it = it;
        isl.idx = idx;
        isl.L = L;
        isl.qstart = qstart;
        isl.n = n;
        isl.done = 0;
      }
      mbar_arrive(&bars->islot_full[qb]);  // every lane, after its own writes
    }
  } else if (warp == 1) {
    // ================================================================ MMA issuer
    if (lane == 0) {
      int g = 0, it_cnt = -1;
      int pend = -1, pend_item = 0;  // tile whose P.V is still to be issued, and its item count
      int last_s = -1, last_pv = -1;  // the last S and P.V issued
      // descriptors of stage 0 / buffer 0; others are offsets of these
      const uint64_t dk0 = desc_k(smem_base);
      const uint64_t dv0 = desc_mn(smem_base + kTileBytes);
      const uint64_t dq0 = desc_k(smem_base + Y::kQOff);
      const uint64_t dp0 = desc_k(smem_base + Y::kPOff);
      bool pend_first = false, pend_last = false;
      auto issue_pv = [&]() -> bool {
        const int b = pend & 1, st = pend % Y::kStages, ob = pend_item & 1;
        if (pend_first) {
          // O^T[ob] is about to be overwritten: the epilogue of item pend_item-2 must have read it
          if (!mbar_wait(&bars->o_empty[ob], ((pend_item >> 1) & 1) ^ 1, wc)) return false;
        }
        if (!mbar_wait(&bars->p_full[b], (pend >> 1) & 1, wc)) return false;
        if (!mbar_wait(F8 ? &bars->vc_full[st] : &bars->v_full[st], (pend / Y::kStages) & 1, wc)) return false;
        tc_fence_after();
        const uint64_t dv = desc_add(dv0, st * kStageBytes);
        const uint64_t dp = desc_add(dp0, b * 2 * kQHalf);
#pragma unroll
        for (int kk = 0; kk < kKeys / 16; ++kk)
          umma_bf16(tmem + kOCol + ob * kN, desc_add(dv, kk * 2048), desc_add(dp, (kk >> 2) * kQHalf + (kk & 3) * 32),
                    F8 ? kIdescO16 : kIdescO, (pend_first && kk == 0) ? 0u : 1u);
        umma_commit(&bars->pv_done[b]);
        umma_commit(&bars->kv_empty[st]);
        if (pend_last) umma_commit(&bars->o_full[ob]);
        last_pv = pend;
        pend = -1;
        return true;
      };
      bool ok = true;
      for (;; ++g) {
        const int st = g % Y::kStages;
        uint64_t* const kf = F8 ? &bars->kc_full[st] : &bars->k_full[st];
        const uint32_t kph = (g / Y::kStages) & 1;
        if (pend >= 0) {
          // Whichever comes first: K(g) landed (then S(g), and P.V(pend)
          // after it, as below) or P(pend) written (then P.V(pend) now, which
          // releases its K/V stage to the producers without waiting for K(g)).
          const uint64_t t0 = globaltimer();
          for (uint32_t i = 1;; ++i) {
            if (mbar_test_wait(kf, kph)) break;
            if (mbar_test_wait(&bars->p_full[pend & 1], (pend >> 1) & 1)) {
              ok = issue_pv();
              break;
            }
            if ((i & 63u) == 0 && globaltimer() - t0 > wc.limit_ns) {
              raise_error(wc.err, PKV_DEVERR_TIMEOUT);
              ok = false;
              break;
            }
          }
          if (!ok) break;
        }
        if (!mbar_wait(kf, kph, wc)) {
          ok = false;
          break;
        }
        const int flags = meta[F8 ? (g & 3) : st].flags;
        if (flags & kMetaDone) {
          if (pend >= 0) ok = issue_pv();
          break;
        }
        if (flags & kMetaFirst) ++it_cnt;
        const int b = g & 1;
        if (!mbar_wait(&bars->s_free[b], ((g >> 1) & 1) ^ 1, wc)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint64_t dk = desc_add(dk0, st * kStageBytes);
        const uint64_t dq = desc_add(dq0, (it_cnt & (Y::kQBufs - 1)) * 2 * kQHalf);
#pragma unroll
        for (int kk = 0; kk < 128 / 16; ++kk)
          umma_bf16(tmem + kSCol + b * kN, desc_add(dk, (kk >> 2) * kHalf + (kk & 3) * 32),
                    desc_add(dq, (kk >> 2) * kQHalf + (kk & 3) * 32), F8 ? kIdescS16 : kIdescS, kk > 0 ? 1u : 0u);
        umma_commit(&bars->s_full[b]);
        last_s = g;
        if (pend >= 0 && !issue_pv()) {
          ok = false;
          break;
        }
        pend = g;
        pend_item = it_cnt;
        pend_first = (flags & kMetaFirst) != 0;
        pend_last = (flags & kMetaLast) != 0;
      }
      if (!ok) {
        // leaving early: let the MMAs already issued finish before TMEM is freed
        if (last_s >= 0) mbar_wait(&bars->s_full[last_s & 1], (last_s >> 1) & 1, wc);
        if (last_pv >= 0) mbar_wait(&bars->pv_done[last_pv & 1], (last_pv >> 1) & 1, wc);
      }
    }
    __syncwarp();
  } else if (warp >= 12) {
    // ================================================================ FP8 converters (warps 12-15)
    // Per stage: the staged K codes (and, on an item's first tile, its Q
    // tile, bf16 -> fp16 in place) become the fp16 K tile, then kc_full;
    // the staged V codes become the fp16 V tile, then vc_full.  The stage's
    // fp16 tiles are free: its producer waited for kv_empty before loading.
    if constexpr (F8) {
      const int c = threadIdx.x - 384;
      int it_cnt = -1;
      for (int g = 0;; ++g) {
        const int st = g % Y::kStages;
        const uint32_t ph = (g / Y::kStages) & 1;
        if (!wait_all(&bars->k_full[st], ph, wc)) break;
        const int flags = meta[g & 3].flags;
        if (flags & kMetaDone) {
          mbar_arrive(&bars->kc_full[st]);  // the MMA and softmax warps see the end
          break;
        }
        // the stage's fp16 tiles are free once the P.V of its previous tile is done
        if (!wait_all(&bars->kv_empty[st], ph ^ 1, wc)) break;
        const uint8_t* codes = smem + Y::kStgOff + st * 2 * kCodeTile;
        uint8_t* kd = smem + st * kStageBytes;
        convert_tile(codes, kd, c);
        if (flags & kMetaFirst) {
          ++it_cnt;
          uint4* q = reinterpret_cast<uint4*>(smem + Y::kQOff + (it_cnt & (Y::kQBufs - 1)) * 2 * kQHalf);
          for (int i = c; i < 2 * kQHalf / 16; i += 128) q[i] = bf16x8_to_f16x8(q[i]);
        }
        fence_proxy_async_smem();  // generic-proxy writes, read by the tensor core
        mbar_arrive(&bars->kc_full[st]);
        if (!wait_all(&bars->v_full[st], ph, wc)) break;
        convert_tile(codes + kCodeTile, kd + kTileBytes, c);
        fence_proxy_async_smem();
        mbar_arrive(&bars->vc_full[st]);
        mbar_arrive(&bars->stage_empty[st]);  // both code tiles of the slot read
      }
    }
  } else {
    // ================================================================ softmax / epilogue
    constexpr int kLog = NR == 4 ? 2 : NR == 8 ? 3 : 4;
    const int q4 = warp & 3;
    const int t = q4 * 32 + lane;  // key of the tile (S^T lane) / output column (O^T lane)
    const uint32_t lane_base = tmem + ((uint32_t)(q4 * 32) << 16);
    EpSlot* slots = reinterpret_cast<EpSlot*>(smem + Y::kSlotOff);
    if (warp < 6) {
      // ---------------------------------------------------------- softmax
      // Failures of waits are carried in `pending` (warp-uniform) to the next
      // agreement barrier (barrier 1 over the 4 softmax warps, which also
      // exchanges the row maxima), where all four warps go on or leave.
      const int my_row = lane >> (5 - kLog);  // row this lane holds after a reduction
      const bool row_writer = (lane & ((1 << (5 - kLog)) - 1)) == 0;
      float m_ref[NR], lsum[NR];
      int vis[NR];
#pragma unroll
      for (int r = 0; r < NR; ++r) {
        m_ref[r] = -CUDART_INF_F;
        lsum[r] = 0.f;
        vis[r] = 0;
      }
      Meta mt{};
      int it_cnt = -1;
      bool pending = false;
      for (int g = 0;; ++g) {
        const int st = g % Y::kStages;
        const int mi = F8 ? (g & 3) : st;
        const int b = g & 1;
        float* redb = red + b * 4 * NR;  // [4 warps][NR], double-buffered by tile
        // the stage's K (and metadata) arrived; the stage is not refilled
        // before this tile's P.V, which needs this tile's P from these warps
        bool fail = pending || !wait_all(F8 ? &bars->kc_full[st] : &bars->k_full[st], (g / Y::kStages) & 1, wc);
        const int flags = fail ? 0 : meta[mi].flags;
        const bool done = (flags & kMetaDone) != 0;
        uint32_t sraw[NR];
#pragma unroll
        for (int r = 0; r < NR; ++r) sraw[r] = 0;
        int kbase = 0;
        if (!fail && !done) {
          if (flags & kMetaFirst) {
            mt = meta[mi];
            ++it_cnt;
#pragma unroll
            for (int r = 0; r < NR; ++r) {
              m_ref[r] = -CUDART_INF_F;
              lsum[r] = 0.f;
              const int tok = (mt.row0 + r) / p.G;
              vis[r] = r < mt.nrows ? min(mt.ke, p.causal ? mt.L - mt.n + tok + 1 : mt.L) : 0;
            }
          }
          kbase = meta[mi].kbase;
          fail = !wait_all(&bars->s_full[b], (g >> 1) & 1, wc);
          if (!fail) {
            tc_fence_after();
            tmem_ld_rows<NR>(lane_base + kSCol + b * kN, sraw);
            tmem_wait_ld();
            tc_fence_before();
            mbar_arrive(&bars->s_free[b]);
          }
        }
        // ---- masked logits of this thread's key; row maxima over the tile
        const int key = kbase + t;
        float v[NR], a[NR];
#pragma unroll
        for (int r = 0; r < NR; ++r) {
          v[r] = key < vis[r] ? __uint_as_float(sraw[r]) : -CUDART_INF_F;
          a[r] = v[r];
        }
        const float wmax = xreduce<NR>(a, lane, MaxOp());
        if (row_writer) redb[q4 * NR + my_row] = wmax;
        if (barrier_any(1, 128, fail || done)) {
          // leaving: at the end of the work (nobody failed), tell the epilogue
          if (!barrier_any(1, 128, fail)) {
            const int ob = (it_cnt + 1) & 1;
            if (wait_all(&bars->ml_empty[ob], (((it_cnt + 1) >> 1) & 1) ^ 1, wc)) {
              if (t == 0) slots[ob].done = 1;
              mbar_arrive(&bars->ml_full[ob]);
            }
          }
          break;
        }
        float alpha[NR], m_use[NR];
        bool any_rescale = false;
#pragma unroll
        for (int r = 0; r < NR; ++r) {
          const float mx =
              fmaxf(fmaxf(redb[r], redb[NR + r]), fmaxf(redb[2 * NR + r], redb[3 * NR + r])) * p.scale_log2;
          alpha[r] = 1.f;
          if (mx > m_ref[r] + kRescaleThreshold) {  // false while both are -inf
            alpha[r] = fast_exp2(m_ref[r] - mx);    // 0 when m_ref is -inf
            any_rescale |= m_ref[r] != -CUDART_INF_F;
            m_ref[r] = mx;
          }
          m_use[r] = m_ref[r] == -CUDART_INF_F ? 0.f : m_ref[r];
        }
        any_rescale = any_rescale && !(flags & kMetaFirst);

        // ---- P (bf16) into this tile's P buffer: row r, column t, 128-byte swizzle
        pending = !wait_all(&bars->pv_done[b], ((g >> 1) & 1) ^ 1, wc);  // P.V of tile g-2 is done
        uint8_t* pbuf = smem + Y::kPOff + b * 2 * kQHalf + (t >> 6) * kQHalf;
        const int pchunk = (t & 63) >> 3, pbyte = (t & 7) * 2;
#pragma unroll
        for (int r = 0; r < NR; ++r) {
          const float e = fast_exp2(fmaf(v[r], p.scale_log2, -m_use[r]));
          lsum[r] = fmaf(lsum[r], alpha[r], e);
          if (!pending) {
            if constexpr (F8)
              *reinterpret_cast<__half*>(pbuf + r * 128 + ((pchunk ^ (r & 7)) << 4) + pbyte) = __float2half_rn(e);
            else
              *reinterpret_cast<__nv_bfloat16*>(pbuf + r * 128 + ((pchunk ^ (r & 7)) << 4) + pbyte) =
                  __float2bfloat16_rn(e);
          }
        }
        if (any_rescale && !pending) {
          // O^T must hold every earlier tile's P.V before it is scaled; thread t
          // owns O^T row t (output column t), whose column r belongs to row r
          pending = !wait_all(&bars->pv_done[b ^ 1], ((g - 1) >> 1) & 1, wc);
          if (!pending) {
            tc_fence_after();
            const uint32_t ocol = lane_base + kOCol + (it_cnt & 1) * kN;
            uint32_t o[NR];
            tmem_ld_rows<NR>(ocol, o);
            tmem_wait_ld();
#pragma unroll
            for (int r = 0; r < NR; ++r) o[r] = __float_as_uint(__uint_as_float(o[r]) * alpha[r]);
            tmem_st_rows<NR>(ocol, o);
            tmem_wait_st();
          }
        }
        if (kbase + kKeys > mt.L && !pending) {
          // keys at or past the sequence's end hold arbitrary bits: zero their V
          // rows (after the tile has landed) so that 0 * V stays 0
          pending = !wait_all(F8 ? &bars->vc_full[st] : &bars->v_full[st], (g / Y::kStages) & 1, wc);
          if (!pending && key >= mt.L) {
            uint4* v0 = reinterpret_cast<uint4*>(smem + st * kStageBytes + kTileBytes + t * 128);
            uint4* v1 = reinterpret_cast<uint4*>(smem + st * kStageBytes + kTileBytes + kHalf + t * 128);
#pragma unroll
            for (int c = 0; c < 8; ++c) v0[c] = v1[c] = make_uint4(0, 0, 0, 0);
          }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(&bars->p_full[b]);

        if (!(flags & kMetaLast)) continue;
        // ---- item end: row sums over the 128 key-threads, handed to the epilogue
        float* reds = red + (b ^ 1) * 4 * NR;  // the other buffer of this tile pair
        {
          float c[NR];
#pragma unroll
          for (int r = 0; r < NR; ++r) c[r] = lsum[r];
          const float wsum = xreduce<NR>(c, lane, AddOp());
          if (row_writer) reds[q4 * NR + my_row] = wsum;
        }
        if (barrier_any(1, 128, pending)) break;
        const int ob = it_cnt & 1;
        pending = !wait_all(&bars->ml_empty[ob], ((it_cnt >> 1) & 1) ^ 1, wc);
        if (!pending) {
          EpSlot& es = slots[ob];
#pragma unroll
          for (int r = 0; r < NR; ++r) {
            if (t == r) {
              es.m[r] = m_ref[r];
              es.l[r] = (reds[r] + reds[NR + r]) + (reds[2 * NR + r] + reds[3 * NR + r]);
            }
          }
          if (t == 0) {
            es.mt = mt;
            es.done = 0;
          }
        }
        // reds[] is rewritten two tiles from now; the slot is complete
        if (barrier_any(1, 128, pending)) break;
        mbar_arrive(&bars->ml_full[ob]);
      }
    } else {
      // ---------------------------------------------------------- epilogue
      // Over the 4 epilogue warps, barrier 3: agreement after each wait that
      // decides what they do next; barrier 2: the split tickets' ordering.
      const int d = t;
      int* flag_last = reinterpret_cast<int*>(tmem_slot + 1);
      bool pending = false;
      for (int it_cnt = 0;; ++it_cnt) {
        const int ob = it_cnt & 1;
        const bool fail = pending || !wait_all(&bars->ml_full[ob], (it_cnt >> 1) & 1, wc);
        if (barrier_any(3, 128, fail)) break;
        const EpSlot& es = slots[ob];
        if (es.done) break;
        const Meta mt = es.mt;
        float mrow[NR], lrow[NR];
#pragma unroll
        for (int r = 0; r < NR; ++r) {
          mrow[r] = es.m[r];
          lrow[r] = r < mt.nrows ? es.l[r] : 1.f;
        }
        mbar_arrive(&bars->ml_empty[ob]);
        pending = !wait_all(&bars->o_full[ob], (it_cnt >> 1) & 1, wc);
        uint32_t o[NR];
        if (!pending) {
          tc_fence_after();
          tmem_ld_rows<NR>(lane_base + kOCol + ob * kN, o);
          tmem_wait_ld();
          tc_fence_before();
          mbar_arrive(&bars->o_empty[ob]);
        }
        const int nr = mt.nrows;
        if (mt.part < 0) {
          if (pending) continue;  // leaves at the next agreement
          // The item finishes its rows.  With a merge group it follows a
          // shared prefix, whose partial rows (complete before this kernel
          // started) are folded in: m = max, weights 2^(m_p - m).
          int pre_base = 0, pre_n = 0, pre_stride = 0;
          if (mt.grp >= 0) {
            const MergeGroup gr = load_group(p.groups + mt.grp);
            pre_base = gr.pre_base;
            pre_n = gr.pre_n;
            pre_stride = gr.pre_stride;
          }
#pragma unroll
          for (int r = 0; r < NR; ++r) {
            if (r < nr) {
              float acc = __uint_as_float(o[r]), lt = lrow[r];
              if (pre_n > 0) {
                float M = mrow[r];
                for (int c = 0; c < pre_n; ++c) M = fmaxf(M, __ldcg(&p.part_ml[pre_base + c * pre_stride + r]).x);
                const float Mu = M == -CUDART_INF_F ? 0.f : M;
                const float w0 = fast_exp2(mrow[r] - Mu);
                acc *= w0;
                lt *= w0;
                for (int c = 0; c < pre_n; ++c) {
                  const int slot = pre_base + c * pre_stride + r;
                  const float2 ml = __ldcg(&p.part_ml[slot]);
                  const float wt = fast_exp2(ml.x - Mu);
                  lt = fmaf(wt, ml.y, lt);
                  acc = fmaf(wt, __ldcg(&p.part_acc[(int64_t)slot * 128 + d]), acc);
                }
              }
              const int row = mt.row0 + r;
              const int tok = row / p.G, gh = row - tok * p.G;
              __nv_bfloat16* orow = reinterpret_cast<__nv_bfloat16*>(p.out) +
                                    ((int64_t)(mt.qstart + tok) * p.Hq + (int64_t)mt.kvh * p.G + gh) * 128;
              orow[d] = __float2bfloat16_rn(acc / lt * p.v_scale);
            }
          }
          continue;
        }
        if (!pending) {
#pragma unroll
          for (int r = 0; r < NR; ++r) {
            if (r < nr) {
              p.part_acc[(int64_t)(mt.part + r) * 128 + d] = __uint_as_float(o[r]);
              if (d == r) p.part_ml[mt.part + r] = make_float2(mrow[r], lrow[r]);
            }
          }
        }
        // The split that completes its merge group combines the group's
        // partial rows: m = max m_p, l = sum l_p 2^(m_p - m), O = sum acc_p 2^(m_p - m) / l.
        // Release: the barrier orders every thread's partial writes before
        // thread 0's fence and ticket; acquire: thread 0's fence after the
        // ticket, then the barrier, before anyone reads other splits' rows.
        if (barrier_any(3, 128, pending)) break;
        if (d == 0) {
          __threadfence();
          *flag_last = atomicAdd(p.tickets + mt.grp, 1);
        }
        named_barrier(2, 128);
        const MergeGroup gr = load_group(p.groups + mt.grp);
        if (*flag_last == gr.nsplit - 1) {
          if (d == 0) __threadfence();
          named_barrier(2, 128);
          // the splits' partial rows, then those over the group's shared prefix
          // (written by the tensor-core kernel, which ran before this one)
          const int nparts = gr.nsplit + gr.pre_n;
          auto slot_of = [&](int k, int r) {
            return k < gr.nsplit ? gr.part_base + k * gr.nrows + r : gr.pre_base + (k - gr.nsplit) * gr.pre_stride + r;
          };
#pragma unroll
          for (int r = 0; r < NR; ++r) {
            if (r < gr.nrows) {
              float M = -CUDART_INF_F;
#pragma unroll 8
              for (int k = 0; k < nparts; ++k) M = fmaxf(M, __ldcg(&p.part_ml[slot_of(k, r)]).x);
              const float Mu = M == -CUDART_INF_F ? 0.f : M;
              float lt = 0.f, acc = 0.f;
#pragma unroll 8
              for (int k = 0; k < nparts; ++k) {
                const int slot = slot_of(k, r);
                const float2 ml = __ldcg(&p.part_ml[slot]);
                const float wt = fast_exp2(ml.x - Mu);
                lt = fmaf(wt, ml.y, lt);
                acc = fmaf(wt, __ldcg(&p.part_acc[(int64_t)slot * 128 + d]), acc);
              }
              const int row = gr.row0 + r;
              const int tok = row / p.G, gh = row - tok * p.G;
              __nv_bfloat16* orow = reinterpret_cast<__nv_bfloat16*>(p.out) +
                                    ((int64_t)(mt.qstart + tok) * p.Hq + (int64_t)gr.kvh * p.G + gh) * 128;
              orow[d] = __float2bfloat16_rn(acc / lt * p.v_scale);
            }
          }
        }
        named_barrier(2, 128);  // the flag is rewritten by the next split item
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
  // Beside the tensor-core kernel this grid skipped its wait for it at
  // launch; it waits here instead, before it completes.  The next call's
  // kernels are launched with programmatic serialization and wait only for
  // this grid, so its completion must imply the tensor-core kernel's (which
  // still reads the plan, counters and tickets that the next call rewrites).
  if (p.no_wait && threadIdx.x == 0) pdl_wait();
}

template <int NR, bool F8>
cudaError_t launch_dectc_t(const AttnParams& p, const CUtensorMap& qmap, const CUtensorMap& kmap,
                           const CUtensorMap& vmap, int grid, cudaStream_t s) {
  static unsigned long long done_mask = 0;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!(__atomic_load_n(&done_mask, __ATOMIC_ACQUIRE) & (1ull << dev))) {
    e = cudaFuncSetAttribute(dectc_kernel<NR, F8>, cudaFuncAttributeMaxDynamicSharedMemorySize, Lay<F8>::kSmem);
    if (e != cudaSuccess) return e;
    __atomic_fetch_or(&done_mask, 1ull << dev, __ATOMIC_RELEASE);
  }
  e = launch_pdl(dectc_kernel<NR, F8>, dim3(grid), dim3(Lay<F8>::kThreads), Lay<F8>::kSmem, s, p, qmap, kmap,
                 vmap);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace

cudaError_t launch_dectc(const AttnParams& p, int rows, const CUtensorMap& qmap, const CUtensorMap& kmap,
                         const CUtensorMap& vmap, int grid, cudaStream_t s) {
  if (rows <= 4) return launch_dectc_t<4, false>(p, qmap, kmap, vmap, grid, s);
  if (rows <= 8) return launch_dectc_t<8, false>(p, qmap, kmap, vmap, grid, s);
  return launch_dectc_t<16, false>(p, qmap, kmap, vmap, grid, s);
}

cudaError_t launch_dectc_fp8(const AttnParams& p, int rows, const CUtensorMap& qmap, const CUtensorMap& kmap,
                             const CUtensorMap& vmap, int grid, cudaStream_t s) {
  if (rows <= 4) return launch_dectc_t<4, true>(p, qmap, kmap, vmap, grid, s);
  if (rows <= 8) return launch_dectc_t<8, true>(p, qmap, kmap, vmap, grid, s);
  return cudaErrorInvalidValue;  // more than 8 rows per item: the CUDA-core kernel serves FP8 pools
}

}  // namespace pkv
