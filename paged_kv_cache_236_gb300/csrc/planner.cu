// Device-side work planner: turns (query_start_loc, context_lens) into work
// lists for the attention kernels without a host round trip.
//
// Each sequence s has n_s query tokens at positions L_s - n_s .. L_s - 1; for
// one kv head its rows are the (token, head-in-group) pairs.  Rows are cut
// into units - groups of kDecRows rows for the CUDA-core kernel, or tiles of
// the whole tokens that fit kMmaRows rows for the tensor-core kernel
// (mma_unit_rows = floor(kMmaRows / G) * G) - and a unit's visible keys
// (0 .. L - n + last_token for causal, all L otherwise) are split into
// chunks so that the item count roughly matches the number of resident CTAs
// times a few waves ("split-KV": long contexts and small batches still fill
// the GPU).  Split items write partial (max, sum, unnormalised accumulator)
// rows; the last split of a unit to finish merges them (a ticket per merge
// group, zeroed here).  The partial-row capacity is the workspace's; if a
// plan would not fit, chunks grow until it does.
//
// Items are emitted largest first (eight size classes relative to the
// chunk), so that the attention kernels, which take items in list order,
// end with small ones and finish together.
//
// One CTA.  The unit instances (sequence, row unit, kv head) are numbered
// sequence major, each sequence's units contiguous (per-sequence unit offsets
// in shared memory); each thread walks a contiguous range of that numbering,
// so that a long prefill sequence's many units spread over many threads.
// Each sequence's (L, n) is read from global memory once and kept in shared
// memory.  Per-class totals are summed per thread, per warp (warp
// reductions) and then across warps; each item takes its slot from its
// warp's cursor within its class's range (items ordered by size class;
// within a class in no particular order, which changes no result).  Every
// pass is thus a few shared-memory round trips, not a chain of dependent
// global reads or contended atomics.
//
// Shared prefixes (when the call asks for them): consecutive decode-shaped
// sequences whose block tables start with the same physical blocks read
// those keys once for the whole run ("cascade").  For each run of at least
// kMinGroupSeqs sequences the common prefix (whole 128-key tiles visible to
// every query of the run) becomes tensor-core items over the run's rows
// (their tokens are contiguous in q), split into npre key chunks, each
// writing partial rows; every member's own decode units then start after the
// prefix, always as merge groups, whose merge folds in the prefix partials.
// Those are complete before the decode kernel runs (the tensor-core kernel
// precedes it in the stream).
#include "kv_rows.cuh"
#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace {

constexpr int kThreads = 512;

constexpr int kWarps = kThreads / 32;
constexpr int kClasses = 8;  // item size classes
// per-thread counters: dec classes, mma classes, merge groups, partial rows (dec, mma)
constexpr int kNumCounts = 2 * kClasses + 3;
constexpr int kCntMerge = 2 * kClasses, kCntPartDec = 2 * kClasses + 1, kCntPartMma = 2 * kClasses + 2;

struct SeqDesc {
  int n, L;
  bool valid, mma;
  int rows, unit_rows, units;
  int pre;        // leading keys read by the sequence's prefix group (0: none)
  int pre_rel;    // its rows' first prefix partial row, relative to the group's
  int pre_shape;  // npre << 24 | the group's rows
};

__device__ __forceinline__ SeqDesc describe_base(const PlanParams& p, int s) {
  SeqDesc d;
  const int a = __ldg(p.query_start_loc + s), b = __ldg(p.query_start_loc + s + 1);
  d.L = __ldg(p.context_lens + s);
  d.n = b - a;
  d.valid = a >= 0 && b >= a && (int64_t)b <= p.T && d.n <= d.L && d.L >= 0 &&
            (int64_t)d.L <= (int64_t)p.max_blocks * p.bs;
  d.rows = d.valid ? d.n * p.G : 0;
  d.mma = p.mma_ok && d.rows > p.dec_rows_max;
  d.unit_rows = d.mma ? p.mma_unit_rows : p.dec_unit_rows;
  d.units = (d.rows + d.unit_rows - 1) / d.unit_rows;
  d.pre = 0;
  return d;
}

// (L, n) of sequence s as read once from global memory; n = -1: invalid.
// Kept in shared memory for up to kPlanSmemSeqs sequences, so that the
// planner's later passes do not repeat the dependent global reads.
constexpr int kPlanSmemSeqs = 4096;

__device__ __forceinline__ SeqDesc describe_from(const PlanParams& p, int2 ln) {
  SeqDesc d;
  d.L = ln.x;
  d.valid = ln.y >= 0;
  d.n = d.valid ? ln.y : 0;
  d.rows = d.valid ? d.n * p.G : 0;
  d.mma = p.mma_ok && d.rows > p.dec_rows_max;
  d.unit_rows = d.mma ? p.mma_unit_rows : p.dec_unit_rows;
  d.units = (d.rows + d.unit_rows - 1) / d.unit_rows;
  d.pre = 0;
  return d;
}

// seq_ln: the shared-memory copy of every sequence's (L, n), or nullptr
__device__ __forceinline__ SeqDesc describe(const PlanParams& p, int s, const int2* seq_ln = nullptr) {
  SeqDesc d = seq_ln ? describe_from(p, seq_ln[s]) : describe_base(p, s);
  d.pre_rel = d.pre_shape = 0;
  if (p.cascade) {
    d.pre = p.seq_pre[s];
    d.pre_rel = p.seq_grp[s];
    d.pre_shape = p.seq_tmp[s];
  }
  return d;
}

// Keys a unit must visit: rows [u*unit_rows, ...) of the sequence.
__device__ __forceinline__ int unit_keys(const SeqDesc& d, int u, int G, int causal) {
  const int r1 = min(d.rows, (u + 1) * d.unit_rows);
  const int last_tok = (r1 - 1) / G;
  return causal ? (d.L - d.n + last_tok + 1) : d.L;
}

__device__ __forceinline__ void split_of(int keys, int chunk, int tile, int& nsplit, int& per) {
  int ns = (keys + chunk - 1) / chunk;
  ns = max(1, min(ns, kMaxSplits));
  per = (keys + ns - 1) / ns;
  per = (per + tile - 1) / tile * tile;
  nsplit = max(1, (keys + per - 1) / per);
}

__device__ __forceinline__ int size_class(int keys, int chunk) {
  // 0 = largest (a full chunk), kClasses-1 = smallest
  const int c = (int)((float)(chunk - keys) * (float)kClasses / (float)max(chunk, 1));
  return min(max(c, 0), kClasses - 1);
}

// Block-wide exclusive scan of K ints per thread (in place); totals[] gets the
// sums.  Warp scans with shuffles; then K threads each scan one counter across
// the warps' totals in shared memory.
template <int K>
__device__ void block_scan(int (&v)[K], int (&totals)[K]) {
  __shared__ int warp_tot[kWarps][K];
  __shared__ int sum_tot[K];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int k = 0; k < K; ++k) {
    int x = v[k];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) warp_tot[warp][k] = x;
    v[k] = x - v[k];  // exclusive within the warp
  }
  __syncthreads();
  if (threadIdx.x < K) {
    int run = 0;
    for (int w = 0; w < kWarps; ++w) {
      const int x = warp_tot[w][threadIdx.x];
      warp_tot[w][threadIdx.x] = run;
      run += x;
    }
    sum_tot[threadIdx.x] = run;
  }
  __syncthreads();
#pragma unroll
  for (int k = 0; k < K; ++k) {
    v[k] += warp_tot[warp][k];
    totals[k] = sum_tot[k];
  }
  __syncthreads();
}

// Walks a contiguous range of unit instances i = (seq_off[s] + u) * Hkv +
// kvh: a unit of rows of one sequence and one kv head, numbered sequence
// major, so that the kv heads of one unit are adjacent.
struct UnitIter {
  int i, end, B, Hkv, s, u, kvh;
  SeqDesc d;
  const int2* seq_ln;  // cached (L, n) per sequence, or nullptr
};

__device__ __forceinline__ void iter_seek(UnitIter& t, const PlanParams& p, const int* seq_off) {
  if (t.i >= t.end) return;
  const int j = t.i / t.Hkv;
  t.kvh = t.i - j * t.Hkv;
  int lo = 0, hi = t.B - 1;  // the last sequence whose first unit is <= j
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (seq_off[mid] <= j) lo = mid; else hi = mid - 1;
  }
  t.s = lo;
  t.u = j - seq_off[lo];
  t.d = describe(p, lo, t.seq_ln);
}

__device__ __forceinline__ void iter_next(UnitIter& t, const PlanParams& p, const int* seq_off) {
  ++t.i;
  if (t.i >= t.end) return;
  if (++t.kvh < t.Hkv) return;
  t.kvh = 0;
  if (++t.u < t.d.units) return;
  int s = t.s + 1;  // the next sequence with units
  while (s < t.B && seq_off[s + 1] == seq_off[s]) ++s;
  t.s = s;
  t.u = 0;
  t.d = describe(p, s, t.seq_ln);
}

constexpr int kSearchWarps = 8;  // sequences per CTA of the prefix search

// Shared-prefix search, one warp per sequence s: seq_pre[s] = whole 128-key
// tiles every query of s sees (decode-shaped sequences only, at most
// kMaxPreTiles), and seq_mask[s] = how many leading blocks of s equal those of
// s-1 within both sequences' visible tiles.  The warp compares the two rows
// 32 blocks at a time, all loads in flight together, and takes the first
// difference with a ballot.  Many CTAs, so the rows of all sequences are read
// in about one round trip; it reads only the caller's metadata.
__global__ void __launch_bounds__(kSearchWarps * 32) prefix_search_kernel(PlanParams p) {
  pdl_launch_dependents();  // the planner may start; it waits for this grid before reading its results
  const int lane = threadIdx.x & 31;
  const int s = blockIdx.x * kSearchWarps + (threadIdx.x >> 5);
  if (s < p.B) {
    const int bpt = kMmaTileKeys / p.bs;
    auto vis_tiles = [&](int q) {
      const SeqDesc d = describe_base(p, q);
      return (d.valid && !d.mma && d.n > 0) ? min(kMaxPreTiles, (d.L - d.n) / kMmaTileKeys) : 0;
    };
    const int v = vis_tiles(s);
    const int vp = s >= 1 ? vis_tiles(s - 1) : 0;
    const int lim = min(v, vp) * bpt;  // blocks to compare
    int eq = 0;
    if (lim > 0) {
      const int32_t* prev = p.block_tables + (int64_t)(s - 1) * p.max_blocks;
      const int32_t* cur = prev + p.max_blocks;
      constexpr int kMaxChunks = (kMaxPreTiles * kMmaTileKeys / 8 + 31) / 32;  // block_size >= 8
      int x[kMaxChunks], y[kMaxChunks];
#pragma unroll
      for (int c = 0; c < kMaxChunks; ++c) {
        const int j = c * 32 + lane;
        x[c] = j < lim ? __ldg(prev + j) : 0;
        y[c] = j < lim ? __ldg(cur + j) : 0;
      }
      eq = lim;
#pragma unroll
      for (int c = kMaxChunks - 1; c >= 0; --c) {  // the lowest differing block wins
        const unsigned m = __ballot_sync(0xffffffffu, x[c] != y[c]);
        if (m) eq = c * 32 + __ffs(m) - 1;
      }
      eq = min(eq, lim);
    }
    if (lane == 0) {
      p.seq_pre[s] = v;
      p.seq_mask[s] = (uint32_t)eq;
    }
  }
  // The planner waits for this grid, and the attention kernels for the
  // planner; wait for the predecessor (the K/V write) so that the chain holds.
  pdl_wait();
}

// From the leading blocks each sequence shares with its predecessor
// (prefix_search_kernel), finds the runs of sequences sharing a prefix and
// sizes their prefix work:
// sh_pre = {prefix items, prefix partial rows, groups read once, groups}.
// Leaves, per sequence s: seq_pre[s] (keys read by its group, 0 if none),
// seq_grp[s] (first partial row of its rows in the group's prefix partials,
// relative to their base) and seq_tmp[s] (npre << 24 | the group's rows); and
// pre_groups[] for the prefix items.  Called by the whole block.
__device__ __noinline__ void plan_prefix_groups(const PlanParams p, int* sh_pre) {
  __shared__ int sh_npre;
  const int tid = threadIdx.x, B = p.B;
  const int bpt = kMmaTileKeys / p.bs;  // blocks per tile
  const int per = (B + kThreads - 1) / kThreads;
  const int a0 = min(B, tid * per), a1 = min(B, a0 + per);
  // seq_pre[s]: whole tiles visible to every query of s; seq_mask[s]: leading
  // blocks of s equal to its predecessor's (both from prefix_search_kernel)
  const int* eqb = reinterpret_cast<const int*>(p.seq_mask);
  // (a) runs: a sequence with no leading tile equal to its predecessor's starts one
  auto equal_tiles = [&](int s) { return eqb[s] / bpt; };
  int ng = 0;
  {
    int nl = 0;
    for (int s = a0; s < a1; ++s) nl += equal_tiles(s) == 0;
    int v[1] = {nl}, tot[1];
    block_scan<1>(v, tot);
    int g = v[0] - 1;
    for (int s = a0; s < a1; ++s) {
      if (equal_tiles(s) == 0) {
        ++g;
        PreGroup pg{};
        pg.s0 = s;
        pg.s1 = s;
        pg.pre_tiles = kMaxPreTiles;
        p.pre_groups[g] = pg;
      }
      p.seq_grp[s] = g;
    }
    ng = tot[0];
  }
  __syncthreads();
  for (int s = a0; s < a1; ++s) {
    const int g = p.seq_grp[s], c = equal_tiles(s);
    if (c > 0) atomicMin(&p.pre_groups[g].pre_tiles, c);  // the run's common prefix
    if (s == B - 1 || equal_tiles(s + 1) == 0) p.pre_groups[g].s1 = s;
  }
  __syncthreads();
  // (b) size the prefix work: about one item per SM (target_mma / 2) in all,
  // and at most half the partial rows of the workspace, or none at all
  const int gper = (ng + kThreads - 1) / kThreads;
  const int g0 = min(ng, tid * gper), g1 = min(ng, g0 + gper);
  int rtiles = 0, rows = 0;
  for (int g = g0; g < g1; ++g) {
    PreGroup& pg = p.pre_groups[g];
    pg.rows = (p.query_start_loc[pg.s1 + 1] - p.query_start_loc[pg.s0]) * p.G;
    if (pg.s1 - pg.s0 + 1 < kMinGroupSeqs) continue;
    rtiles += p.Hkv * ((pg.rows + p.mma_unit_rows - 1) / p.mma_unit_rows);
    rows += p.Hkv * pg.rows;
  }
  {
    int v[2] = {rtiles, rows}, tot[2];
    block_scan<2>(v, tot);
    if (tid == 0) {
      // about one wave: the prefix items run before any decode item starts
      int npre = tot[0] > 0 ? max(1, (p.target_mma / 2) / tot[0]) : 0;
      npre = min(npre, kMaxPreTiles);
      while (npre > 0 && (int64_t)tot[1] * npre > p.part_cap / 2) --npre;
      sh_npre = npre;
    }
    __syncthreads();
  }
  const int npre = sh_npre;
  int nitems = 0, nrows = 0, nvalid = 0;
  for (int g = g0; g < g1; ++g) {
    PreGroup& pg = p.pre_groups[g];
    pg.valid = npre > 0 && pg.s1 - pg.s0 + 1 >= kMinGroupSeqs && pg.pre_tiles >= 1;
    if (pg.valid) {
      const int chunk_tiles = (pg.pre_tiles + min(npre, pg.pre_tiles) - 1) / min(npre, pg.pre_tiles);
      pg.npre = (pg.pre_tiles + chunk_tiles - 1) / chunk_tiles;
      nitems += p.Hkv * ((pg.rows + p.mma_unit_rows - 1) / p.mma_unit_rows) * pg.npre;
      nrows += p.Hkv * pg.rows * pg.npre;
      ++nvalid;
    } else {
      pg.npre = 0;
    }
  }
  {
    int v[3] = {nitems, nrows, nvalid}, tot[3];
    block_scan<3>(v, tot);
    int io = v[0], ro = v[1];
    for (int g = g0; g < g1; ++g) {
      PreGroup& pg = p.pre_groups[g];
      pg.item_off = io;
      pg.part_off = ro;
      if (pg.valid) {
        io += p.Hkv * ((pg.rows + p.mma_unit_rows - 1) / p.mma_unit_rows) * pg.npre;
        ro += p.Hkv * pg.rows * pg.npre;
      }
    }
    if (tid == 0) {
      sh_pre[0] = tot[0];
      sh_pre[1] = tot[1];
      sh_pre[2] = tot[2];
      sh_pre[3] = ng;
    }
  }
  __syncthreads();
  // (c) each member's suffix starts after its group's prefix; where its rows'
  // prefix partials are
  for (int s = a0; s < a1; ++s) {
    const PreGroup pg = p.pre_groups[p.seq_grp[s]];
    p.seq_pre[s] = pg.valid ? pg.pre_tiles * kMmaTileKeys : 0;
    p.seq_grp[s] = pg.valid ? pg.part_off + (p.query_start_loc[s] - p.query_start_loc[pg.s0]) * p.G : 0;
    p.seq_tmp[s] = pg.valid ? (pg.npre << 24) | pg.rows : 0;
  }
  __syncthreads();
}

// CTAs 1 .. write_ctas of the planner's grid: the step's new K/V rows, one
// warp per token, after the predecessor grid has completed (stream order:
// the previous call's kernels may still read the pool).  The attention
// kernels wait for this whole grid, so they see these rows and the plan.
__device__ __noinline__ void write_new_rows(const PlanParams& p) {
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int64_t warps = (int64_t)(gridDim.x - 1) * (kThreads / 32);
  for (int64_t t = (int64_t)(blockIdx.x - 1) * (kThreads / 32) + (threadIdx.x >> 5); t < p.wT; t += warps) {
    if (p.write_mode == 1) {
      if (p.w_row <= 64)
        copy_token_rows<2>(static_cast<const uint8_t*>(p.wk), static_cast<const uint8_t*>(p.wv), p.wslots,
                           static_cast<uint8_t*>(p.wkc), static_cast<uint8_t*>(p.wvc), t, p.w_num_slots, p.w_row,
                           p.wk_stride, p.wv_stride, p.err, lane);
      else
        copy_token_rows<4>(static_cast<const uint8_t*>(p.wk), static_cast<const uint8_t*>(p.wv), p.wslots,
                           static_cast<uint8_t*>(p.wkc), static_cast<uint8_t*>(p.wvc), t, p.w_num_slots, p.w_row,
                           p.wk_stride, p.wv_stride, p.err, lane);
    } else if (p.write_mode == 2) {
      quantize_token_rows<uint16_t>(static_cast<const uint16_t*>(p.wk), static_cast<const uint16_t*>(p.wv), p.wslots,
                                    static_cast<uint8_t*>(p.wkc), static_cast<uint8_t*>(p.wvc), t, p.w_num_slots,
                                    p.w_row, p.wk_stride, p.wv_stride, p.wk_scale, p.wv_scale, p.err, lane);
    } else {
      quantize_token_rows<float>(static_cast<const float*>(p.wk), static_cast<const float*>(p.wv), p.wslots,
                                 static_cast<uint8_t*>(p.wkc), static_cast<uint8_t*>(p.wvc), t, p.w_num_slots,
                                 p.w_row, p.wk_stride, p.wv_stride, p.wk_scale, p.wv_scale, p.err, lane);
    }
  }
}

__global__ void __launch_bounds__(kThreads, 1) plan_kernel(PlanParams p) {
  // The attention kernel may start its prologue while this plans (it waits
  // for this grid).  This grid may start while its predecessor runs: the
  // predecessors that let it (paged_kv_write, the shared-prefix search)
  // write neither the metadata read here nor anything written here, so the
  // plan is computed at once and the wait for the predecessor comes before
  // the first write that later kernels read (which also makes this grid's
  // completion imply the predecessor's, as the attention kernels need).
  // With a fused write, CTAs 1 .. write_ctas write the step's new K/V rows
  // (after the same wait) while CTA 0 plans.
  pdl_launch_dependents();
  if (blockIdx.x > 0) {  // the step's new K/V rows (a fused write)
    write_new_rows(p);
    return;
  }
  extern __shared__ int seq_off[];  // [B + 1]: first unit of each sequence (per kv head)
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int B = p.B;
  // after seq_off (8-byte aligned): every sequence's (L, n) when B <= kPlanSmemSeqs
  int2* const seq_ln = B <= kPlanSmemSeqs ? reinterpret_cast<int2*>(seq_off + ((B + 2) & ~1)) : nullptr;

  // ---- shared-prefix groups
  __shared__ int sh_pre[4];  // prefix items, prefix partial rows, groups read once, groups
  if (tid == 0) sh_pre[0] = sh_pre[1] = sh_pre[2] = sh_pre[3] = 0;
  __syncthreads();
  if (p.cascade) {
    pdl_wait();  // the shared-prefix search (the predecessor) is complete
    plan_prefix_groups(p, sh_pre);
  }

  // ---- units per sequence (invalid sequences: none; their rows are zeroed below)
  bool any_invalid = false;
  for (int s = tid; s < B; s += kThreads) {
    const SeqDesc d = describe(p, s);
    any_invalid |= !d.valid;
    seq_off[s] = d.units;  // 0 for an invalid sequence
    if (seq_ln) seq_ln[s] = make_int2(d.L, d.valid ? d.n : -1);
  }
  __syncthreads();
  {
    // exclusive scan of seq_off[0 .. B) in place; seq_off[B] = units per kv head
    const int per = (B + kThreads - 1) / kThreads;
    const int s0 = min(B, tid * per), s1 = min(B, s0 + per);
    int sum = 0;
    for (int s = s0; s < s1; ++s) sum += seq_off[s];
    int v[1] = {sum}, tot[1];
    block_scan<1>(v, tot);
    int run = v[0];
    for (int s = s0; s < s1; ++s) {
      const int x = seq_off[s];
      seq_off[s] = run;
      run += x;
    }
    if (tid == 0) seq_off[B] = tot[0];
    __syncthreads();
  }
  const int U = seq_off[B];
  const int N = U * p.Hkv;  // unit instances
  const int per_thread = (N + kThreads - 1) / kThreads;
  const int i0 = min(N, tid * per_thread), i1 = min(N, i0 + per_thread);

  // ---- total keys per path, for the chunk sizes
  __shared__ unsigned long long sh_wsum[kWarps][2];
  __shared__ int sh_chunk[2];
  __shared__ int sh_mma_ctas;
  __shared__ int sh_state;
  unsigned long long w_dec = 0, w_mma = 0;
  {
    UnitIter t{i0, i1, B, p.Hkv, 0, 0, 0, {}, seq_ln};
    for (iter_seek(t, p, seq_off); t.i < t.end; iter_next(t, p, seq_off))
      (t.d.mma ? w_mma : w_dec) += (unsigned long long)(unit_keys(t.d, t.u, p.G, p.causal) - t.d.pre);
  }
  // warp sums, then one thread adds the warps' (no contended 64-bit atomics)
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    w_dec += __shfl_xor_sync(0xffffffffu, w_dec, o);
    w_mma += __shfl_xor_sync(0xffffffffu, w_mma, o);
  }
  if ((tid & 31) == 0) {
    sh_wsum[tid >> 5][0] = w_dec;
    sh_wsum[tid >> 5][1] = w_mma;
  }
  __syncthreads();
  if (tid == 0) {
    unsigned long long wd = 0, wm = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      wd += sh_wsum[w][0];
      wm += sh_wsum[w][1];
    }
    // Side by side: the tensor-core items (compute-bound) on mma_ctas SMs,
    // the decode items (HBM-bound) on the rest, both at once, the split
    // balancing a time model measured on this GPU: ~10 ns per (128-row unit,
    // key) on one SM for the former (x1.15 for its coarse items' tail); for
    // the latter the K+V bytes at 6.5 TB/s in all, at most 60 GB/s per SM.
    int mma_ctas = p.sms;
    if (p.side_by_side && wd > 0 && wm > 0) {
      const float tm1 = (float)wm * 1.0e-2f * 1.15f;  // µs on one SM
      const float db = (float)wd * (float)p.kv_key_bytes;
      const float btot = 6.5e6f, bsm = 6.0e4f;  // bytes per µs
      auto dec_us = [&](int n) { return db / fminf(btot, (float)n * bsm); };
      auto total = [&](int k) { return fmaxf(tm1 / (float)k, dec_us(p.sms - k)); };
      float best = tm1 / (float)p.sms + dec_us(p.sms);  // one after the other
      // the optimum balances the two sides: where the decode side is
      // HBM-bound (k1) or bound by its SMs (k2); try the integers around both
      const int k1 = (int)ceilf(tm1 * btot / db);
      const int k2 = (int)(tm1 * (float)p.sms * bsm / (db + tm1 * bsm));
      const int cand[5] = {k1 - 1, k1, k2, k2 + 1, k2 + 2};
      for (int c = 0; c < 5; ++c) {
        const int k = min(max(cand[c], 1), p.sms - 1);
        const float t = total(k);
        if (t < best) {
          best = t;
          mma_ctas = k;
        }
      }
    }
    sh_mma_ctas = mma_ctas;
    const int tgt_dec = mma_ctas < p.sms ? max(1, p.target_dec * (p.sms - mma_ctas) / p.sms) : p.target_dec;
    const int tgt_mma = max(1, p.target_mma * mma_ctas / max(1, p.sms));
    unsigned long long cd = (wd + tgt_dec - 1) / (unsigned long long)tgt_dec;
    unsigned long long cm = (wm + tgt_mma - 1) / (unsigned long long)tgt_mma;
    cd = max(cd, (unsigned long long)p.min_chunk_dec);
    cm = max(cm, (unsigned long long)p.min_chunk_mma);
    cd = (cd + p.dec_tile_keys - 1) / p.dec_tile_keys * p.dec_tile_keys;
    cm = (cm + kMmaTileKeys - 1) / kMmaTileKeys * kMmaTileKeys;
    sh_chunk[0] = (int)min(cd, (unsigned long long)(1 << 30));
    sh_chunk[1] = (int)min(cm, (unsigned long long)(1 << 30));
  }
  __syncthreads();

  // ---- count items per size class, merge groups and partial rows; grow the
  // chunks until the plan fits the workspace.  Totals go through shared
  // atomics; an item's slot is taken from its class's cursor when it is
  // written (the order within a class does not change any result: every
  // item computes the same rows whichever CTA takes it, and split merges
  // follow split order).
  // Counts are kept per thread in registers, summed per warp with warp
  // reductions (no contended shared atomics), then across warps; each warp's
  // exclusive base per counter is what its threads' items start from when
  // emitted (the same threads walk the same instances in both passes).
  __shared__ int s_tot[kNumCounts];
  __shared__ int s_cur[kNumCounts];           // class offsets (largest class first)
  __shared__ int s_wcnt[kWarps][kNumCounts];  // per-warp counts, then per-warp bases
  __shared__ int s_wcur[kWarps][kNumCounts];  // per-warp emit cursors
  for (int iter = 0;; ++iter) {
    const int cd = sh_chunk[0], cm = sh_chunk[1];
    int cnt[kNumCounts];
#pragma unroll
    for (int k = 0; k < kNumCounts; ++k) cnt[k] = 0;
    auto add = [&](int idx, int v) {
#pragma unroll
      for (int k = 0; k < kNumCounts; ++k) cnt[k] += idx == k ? v : 0;
    };
    {
      UnitIter t{i0, i1, B, p.Hkv, 0, 0, 0, {}, seq_ln};
      for (iter_seek(t, p, seq_off); t.i < t.end; iter_next(t, p, seq_off)) {
        const SeqDesc& d = t.d;
        const int chunk = d.mma ? cm : cd;
        const int cb = d.mma ? kClasses : 0;
        const int keys = unit_keys(d, t.u, p.G, p.causal) - d.pre;
        int ns, per;
        split_of(keys, chunk, d.mma ? kMmaTileKeys : p.dec_tile_keys, ns, per);
        if (ns > 1) add(cb + size_class(per, chunk), ns - 1);  // all splits but the last are full
        add(cb + size_class(keys - (ns - 1) * per, chunk), 1);
        if (ns > 1 || d.pre > 0) {
          add(kCntMerge, 1);
          if (ns > 1) add(d.mma ? kCntPartMma : kCntPartDec, ns * min(d.rows - t.u * d.unit_rows, d.unit_rows));
        }
      }
    }
#pragma unroll
    for (int k = 0; k < kNumCounts; ++k) {
      const int v = __reduce_add_sync(0xffffffffu, cnt[k]);
      if (lane == 0) s_wcnt[warp][k] = v;
    }
    __syncthreads();
    if (tid < kNumCounts) {
      int tot = 0;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) tot += s_wcnt[w][tid];
      s_tot[tid] = tot;
    }
    __syncthreads();
    if (tid == 0) {
      int nd = 0, nm = 0;
#pragma unroll
      for (int k = 0; k < kClasses; ++k) {
        nd += s_tot[k];
        nm += s_tot[kClasses + k];
      }
      const int pd = s_tot[kCntPartDec], pm = s_tot[kCntPartMma];
      const bool fits = nd <= p.dec_cap && nm + sh_pre[0] <= p.mma_cap && s_tot[kCntMerge] <= p.merge_cap &&
                        (int64_t)pd + pm + sh_pre[1] <= p.part_cap;
      sh_state = fits ? 1 : 0;
      // Once: if the decode items are mostly full chunks (long sequences
      // split) and leave a last wave less than half full, grow the chunk so
      // that the count drops to whole waves.  Items of mixed sizes are left
      // to the largest-first order.
      const int P = max(1, sh_mma_ctas < p.sms ? p.dec_ctas * (p.sms - sh_mma_ctas) / p.sms : p.dec_ctas);
      const int extra = nd % P;
      if (fits && iter == 0 && nd > P && extra > 0 && 2 * extra <= P && 4 * s_tot[0] >= 3 * nd) {
        const long long grown = ((long long)cd * nd + (nd - extra) - 1) / (nd - extra);
        sh_chunk[0] = (int)min((grown + p.dec_tile_keys - 1) / p.dec_tile_keys * p.dec_tile_keys, (long long)(1 << 30));
        sh_state = 0;
      }
      if (!fits) {
        if (iter >= 40) {
          raise_error(p.err, PKV_DEVERR_PLAN_OVERFLOW);
          sh_state = 2;
        }
        const bool dec_over = nd > p.dec_cap || pd >= pm;
        const bool mma_over = nm > p.mma_cap || pm > pd;
        if (dec_over) sh_chunk[0] = (int)min(2LL * cd, (long long)(1 << 30));
        if (mma_over) sh_chunk[1] = (int)min(2LL * cm, (long long)(1 << 30));
      }
      if (sh_state == 1) {
        // cursors: class k's items start after all larger classes' (largest first)
        int od = 0, om = 0;
#pragma unroll
        for (int k = 0; k < kClasses; ++k) {
          s_cur[k] = od;
          od += s_tot[k];
          s_cur[kClasses + k] = om;
          om += s_tot[kClasses + k];
        }
        s_cur[kCntMerge] = 0;
        s_cur[kCntPartDec] = 0;  // partial rows of both kinds from one range
        s_cur[kCntPartMma] = 0;
      }
    }
    __syncthreads();
    if (sh_state) break;
  }
  // per-warp bases: warp w's items of counter k start after those of warps
  // 0 .. w-1 (partial rows of both kinds share one range)
  if (tid < kNumCounts && tid != kCntPartMma) {
    int run = 0;
    for (int w = 0; w < kWarps; ++w) {
      const int c = s_wcnt[w][tid] + (tid == kCntPartDec ? s_wcnt[w][kCntPartMma] : 0);
      s_wcnt[w][tid] = run;
      s_wcur[w][tid] = 0;
      run += c;
    }
  }
  __syncthreads();
  if (sh_state == 2) {  // cannot happen with capacities from workspace_layout; emit nothing
    pdl_wait();
    if (tid == 0) {
      p.header->n_dec = 0;
      p.header->n_mma = 0;
      p.header->mma_ctas = p.sms;
      p.header->n_merge = 0;
    }
    return;
  }

  pdl_wait();
  if (any_invalid) {  // zero the addressable rows of this thread's invalid sequences
    for (int s = tid; s < B; s += kThreads) {
      if (describe_base(p, s).valid) continue;
      raise_error(p.err, PKV_DEVERR_BAD_SEQUENCE);
      const int a = p.query_start_loc[s], b = p.query_start_loc[s + 1];
      if (a >= 0 && b > a && (int64_t)b <= p.T) {
        int4* o = reinterpret_cast<int4*>(static_cast<uint8_t*>(p.out) + (int64_t)a * p.out_row_bytes);
        const int64_t n16 = (int64_t)(b - a) * p.out_row_bytes / 16;
        for (int64_t i = 0; i < n16; ++i) o[i] = make_int4(0, 0, 0, 0);
      }
    }
  }

  // ---- emit
  const int cd = sh_chunk[0], cm = sh_chunk[1];
  const int pre_part_base = s_tot[kCntPartDec] + s_tot[kCntPartMma];  // prefix partial rows follow the units'
  {
    UnitIter t{i0, i1, B, p.Hkv, 0, 0, 0, {}, seq_ln};
    for (iter_seek(t, p, seq_off); t.i < t.end; iter_next(t, p, seq_off)) {
      const SeqDesc& d = t.d;
      const int s = t.s, u = t.u, kvh = t.kvh;
      WorkItem* items = d.mma ? p.mma_items : p.dec_items;
      const int chunk = d.mma ? cm : cd;
      const int cbase = d.mma ? kClasses : 0;
      const int kend = unit_keys(d, u, p.G, p.causal);
      const int keys = kend - d.pre;
      const int r0 = u * d.unit_rows;
      const int nr = min(d.rows - r0, d.unit_rows);
      int ns, per;
      split_of(keys, chunk, d.mma ? kMmaTileKeys : p.dec_tile_keys, ns, per);
      int grp = -1, part_base = 0;
      if (ns > 1 || d.pre > 0) {
        // A unit after a shared prefix always names a merge group (where its
        // prefix partials are); unsplit, its one item folds them in itself.
        grp = s_wcnt[warp][kCntMerge] + atomicAdd(&s_wcur[warp][kCntMerge], 1);
        if (ns > 1) part_base = s_wcnt[warp][kCntPartDec] + atomicAdd(&s_wcur[warp][kCntPartDec], ns * nr);
        MergeGroup g;
        g.seq = s;
        g.kvh = kvh;
        g.row0 = r0;
        g.nrows = nr;
        g.nsplit = ns;
        g.part_base = part_base;
        g.pre_base = 0;
        g.pre_n = 0;
        g.pre_stride = 0;
        g.pad0 = g.pad1 = g.pad2 = 0;
        if (d.pre > 0) {
          // this unit's rows in its group's prefix partials ([kvh][chunk][row])
          const int npre = d.pre_shape >> 24, grows = d.pre_shape & 0xffffff;
          g.pre_base = pre_part_base + d.pre_rel + kvh * npre * grows + r0;
          g.pre_n = npre;
          g.pre_stride = grows;
        }
        p.merges[grp] = g;
        p.tickets[grp] = 0;
      }
      const int full_cls = cbase + size_class(per, chunk);
      const int last_cls = cbase + size_class(keys - (ns - 1) * per, chunk);
      const int full0 =
          ns > 1 ? s_cur[full_cls] + s_wcnt[warp][full_cls] + atomicAdd(&s_wcur[warp][full_cls], ns - 1) : 0;
      const int last0 = s_cur[last_cls] + s_wcnt[warp][last_cls] + atomicAdd(&s_wcur[warp][last_cls], 1);
      for (int sp = 0; sp < ns; ++sp) {
        WorkItem it;
        it.seq = s;
        it.kvh = kvh;
        it.row0 = r0;
        it.nrows = nr;
        it.kb = d.pre + sp * per;
        it.ke = min(kend, d.pre + (sp + 1) * per);
        it.part = ns > 1 ? part_base + sp * nr : -1;
        it.grp = grp;
        items[sp == ns - 1 ? last0 : full0 + sp] = it;
      }
    }
  }
  // ---- prefix items, after the other tensor-core items
  if (sh_pre[0] > 0) {
    int nm = 0;
#pragma unroll
    for (int k = 0; k < kClasses; ++k) nm += s_tot[kClasses + k];
    const int ng = sh_pre[3];
    // item k of a group: kv head, row tile, key chunk (chunk fastest)
    auto emit = [&](const PreGroup& pg, int k) {
      const int rt = (pg.rows + p.mma_unit_rows - 1) / p.mma_unit_rows;
      const int per_keys = (pg.pre_tiles + pg.npre - 1) / pg.npre * kMmaTileKeys;
      const int c = k % pg.npre, t = (k / pg.npre) % rt, kvh = k / (pg.npre * rt);
      WorkItem it;
      it.seq = pg.s0;  // the group's rows are its tokens onwards
      it.kvh = kvh;
      it.row0 = t * p.mma_unit_rows;
      it.nrows = min(p.mma_unit_rows, pg.rows - it.row0);
      it.kb = c * per_keys;
      it.ke = min(pg.pre_tiles * kMmaTileKeys, (c + 1) * per_keys);
      it.part = pre_part_base + pg.part_off + (kvh * pg.npre + c) * pg.rows + it.row0;
      it.grp = -1;  // merged by the decode kernel, with the members' own keys
      p.mma_items[nm + pg.item_off + k] = it;
    };
    if (ng <= 64) {  // few groups: all threads share out each group's items
      for (int g = 0; g < ng; ++g) {
        const PreGroup pg = p.pre_groups[g];
        if (!pg.valid) continue;
        const int n = p.Hkv * ((pg.rows + p.mma_unit_rows - 1) / p.mma_unit_rows) * pg.npre;
        for (int k = tid; k < n; k += kThreads) emit(pg, k);
      }
    } else {
      for (int g = tid; g < ng; g += kThreads) {
        const PreGroup pg = p.pre_groups[g];
        if (!pg.valid) continue;
        const int n = p.Hkv * ((pg.rows + p.mma_unit_rows - 1) / p.mma_unit_rows) * pg.npre;
        for (int k = 0; k < n; ++k) emit(pg, k);
      }
    }
  }
  if (tid == 0) {
    int nd = 0, nm = 0;
#pragma unroll
    for (int k = 0; k < kClasses; ++k) {
      nd += s_tot[k];
      nm += s_tot[kClasses + k];
    }
    p.header->n_dec = nd;
    p.header->n_mma = nm + sh_pre[0];
    p.header->n_pre = sh_pre[0];
    p.header->n_groups = sh_pre[2];
    p.header->n_merge = s_tot[kCntMerge];
    p.header->chunk_dec = cd;
    p.header->chunk_mma = cm;
    p.header->part_rows = s_tot[kCntPartDec] + s_tot[kCntPartMma] + sh_pre[1];
    p.header->dec_counter = 0;
    p.header->mma_counter = 0;
    p.header->merge_counter = 0;
    p.header->mma_ctas = sh_mma_ctas;
  }
}

}  // namespace

cudaError_t launch_prefix_search(const PlanParams& p, cudaStream_t s) {
  if (p.B <= 0) return cudaSuccess;
  const cudaError_t e = launch_pdl(prefix_search_kernel, dim3((p.B + kSearchWarps - 1) / kSearchWarps),
                                   dim3(kSearchWarps * 32), 0, s, p);
  return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_planner(const PlanParams& p, cudaStream_t s) {
  const size_t smem = (size_t)((p.B + 2) & ~1) * sizeof(int) + (p.B <= kPlanSmemSeqs ? (size_t)p.B * sizeof(int2) : 0);
  if (p.B > kMaxPlanSeqs) return cudaErrorInvalidValue;
  static unsigned long long done_mask = 0;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!(__atomic_load_n(&done_mask, __ATOMIC_ACQUIRE) & (1ull << dev))) {
    const size_t most = ((kMaxPlanSeqs + 2) & ~1) * sizeof(int);  // seq_off alone, above kPlanSmemSeqs
    static_assert(((kPlanSmemSeqs + 2) & ~1) * sizeof(int) + kPlanSmemSeqs * sizeof(int2) <=
                      ((kMaxPlanSeqs + 2) & ~1) * sizeof(int),
                  "planner shared memory");
    e = cudaFuncSetAttribute(plan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)most);
    if (e != cudaSuccess) return e;
    __atomic_fetch_or(&done_mask, 1ull << dev, __ATOMIC_RELEASE);
  }
  e = launch_pdl(plan_kernel, dim3(1 + p.write_ctas), dim3(kThreads), smem, s, p);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace pkv
