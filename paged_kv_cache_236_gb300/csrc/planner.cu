// Device-side work planner: turns (query_start_loc, context_lens) into work
// lists for the attention kernels without a host round trip.
//
// Each sequence s has n_s query tokens at positions L_s - n_s .. L_s - 1; for
// one kv head its rows are the (token, head-in-group) pairs.  Rows are cut
// into units - groups of kDecRows rows for the CUDA-core kernel, or tiles of
// kMmaRows rows for the tensor-core kernel - and a unit's visible keys
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
// One CTA.  The unit instances (kv head, sequence, row unit) are numbered
// kv head major, each sequence's units contiguous (per-sequence unit offsets
// in shared memory); each thread walks a contiguous range of that numbering,
// so that a long prefill sequence's many units spread over many threads.
// Block-wide exclusive scans give every item a fixed slot (items ordered by
// size class, then unit instance, then split).
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
};

__device__ __forceinline__ SeqDesc describe(const PlanParams& p, int s) {
  SeqDesc d;
  const int a = __ldg(p.query_start_loc + s), b = __ldg(p.query_start_loc + s + 1);
  d.L = __ldg(p.context_lens + s);
  d.n = b - a;
  d.valid = a >= 0 && b >= a && (int64_t)b <= p.T && d.n <= d.L && d.L >= 0 &&
            (int64_t)d.L <= (int64_t)p.max_blocks * p.bs;
  d.rows = d.valid ? d.n * p.G : 0;
  d.mma = p.mma_ok && d.rows > p.dec_rows_max;
  d.unit_rows = d.mma ? kMmaRows : p.dec_unit_rows;
  d.units = (d.rows + d.unit_rows - 1) / d.unit_rows;
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

// Walks a contiguous range of unit instances i = kvh * U + seq_off[s] + u.
struct UnitIter {
  int i, end, U, B, kvh, s, u;
  SeqDesc d;
};

__device__ __forceinline__ void iter_seek(UnitIter& t, const PlanParams& p, const int* seq_off) {
  if (t.i >= t.end) return;
  t.kvh = t.i / t.U;
  const int j = t.i - t.kvh * t.U;
  int lo = 0, hi = t.B - 1;  // the last sequence whose first unit is <= j
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (seq_off[mid] <= j) lo = mid; else hi = mid - 1;
  }
  t.s = lo;
  t.u = j - seq_off[lo];
  t.d = describe(p, lo);
}

__device__ __forceinline__ void iter_next(UnitIter& t, const PlanParams& p, const int* seq_off) {
  ++t.i;
  if (t.i >= t.end) return;
  if (++t.u < t.d.units) return;
  // next sequence with units (or the next kv head's first one)
  int s = t.s + 1;
  while (s < t.B && seq_off[s + 1] == seq_off[s]) ++s;
  if (s >= t.B) {
    ++t.kvh;
    s = 0;
    while (seq_off[s + 1] == seq_off[s]) ++s;
  }
  t.s = s;
  t.u = 0;
  t.d = describe(p, s);
}

__global__ void __launch_bounds__(kThreads, 1) plan_kernel(PlanParams p) {
  // The attention kernel may start its prologue while this plans (it waits
  // for this grid).  This grid waits for its own predecessor before reading
  // the metadata, which that predecessor may have produced.
  pdl_launch_dependents();
  pdl_wait();
  extern __shared__ int seq_off[];  // [B + 1]: first unit of each sequence (per kv head)
  const int tid = threadIdx.x;
  const int B = p.B;

  // ---- units per sequence; zero the rows of invalid sequences
  for (int s = tid; s < B; s += kThreads) {
    const SeqDesc d = describe(p, s);
    if (!d.valid) {
      raise_error(p.err, PKV_DEVERR_BAD_SEQUENCE);
      const int a = p.query_start_loc[s], b = p.query_start_loc[s + 1];
      if (a >= 0 && b > a && (int64_t)b <= p.T) {  // zero the rows that are addressable
        int4* o = reinterpret_cast<int4*>(static_cast<uint8_t*>(p.out) + (int64_t)a * p.out_row_bytes);
        const int64_t n16 = (int64_t)(b - a) * p.out_row_bytes / 16;
        for (int64_t i = 0; i < n16; ++i) o[i] = make_int4(0, 0, 0, 0);
      }
    }
    seq_off[s] = d.units;  // 0 for an invalid sequence
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
  __shared__ int sh_state;
  unsigned long long w_dec = 0, w_mma = 0;
  {
    UnitIter t{i0, i1, U, B, 0, 0, 0, {}};
    for (iter_seek(t, p, seq_off); t.i < t.end; iter_next(t, p, seq_off))
      (t.d.mma ? w_mma : w_dec) += (unsigned long long)unit_keys(t.d, t.u, p.G, p.causal);
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
    unsigned long long cd = (wd + p.target_dec - 1) / (unsigned long long)max(1, p.target_dec);
    unsigned long long cm = (wm + p.target_mma - 1) / (unsigned long long)max(1, p.target_mma);
    cd = max(cd, (unsigned long long)p.min_chunk_dec);
    cm = max(cm, (unsigned long long)p.min_chunk_mma);
    cd = (cd + p.dec_tile_keys - 1) / p.dec_tile_keys * p.dec_tile_keys;
    cm = (cm + kMmaTileKeys - 1) / kMmaTileKeys * kMmaTileKeys;
    sh_chunk[0] = (int)min(cd, (unsigned long long)(1 << 30));
    sh_chunk[1] = (int)min(cm, (unsigned long long)(1 << 30));
  }
  __syncthreads();

  // ---- count items per size class, merge groups and partial rows; grow the
  // chunks until the plan fits the workspace
  __shared__ int s_cnt[kNumCounts][kThreads];  // per-thread counters, then running offsets
  int cnt[kNumCounts], tot[kNumCounts];
  for (int iter = 0;; ++iter) {
    const int cd = sh_chunk[0], cm = sh_chunk[1];
#pragma unroll
    for (int k = 0; k < kNumCounts; ++k) s_cnt[k][tid] = 0;
    UnitIter t{i0, i1, U, B, 0, 0, 0, {}};
    for (iter_seek(t, p, seq_off); t.i < t.end; iter_next(t, p, seq_off)) {
      const SeqDesc& d = t.d;
      const int chunk = d.mma ? cm : cd;
      const int cb = d.mma ? kClasses : 0;
      const int keys = unit_keys(d, t.u, p.G, p.causal);
      int ns, per;
      split_of(keys, chunk, d.mma ? kMmaTileKeys : p.dec_tile_keys, ns, per);
      s_cnt[cb + size_class(per, chunk)][tid] += ns - 1;  // all splits but the last are full
      s_cnt[cb + size_class(keys - (ns - 1) * per, chunk)][tid] += 1;
      if (ns > 1) {
        s_cnt[kCntMerge][tid] += 1;
        s_cnt[d.mma ? kCntPartMma : kCntPartDec][tid] += ns * min(d.rows - t.u * d.unit_rows, d.unit_rows);
      }
    }
#pragma unroll
    for (int k = 0; k < kNumCounts; ++k) cnt[k] = s_cnt[k][tid];
    block_scan<kNumCounts>(cnt, tot);
    if (tid == 0) {
      int nd = 0, nm = 0;
#pragma unroll
      for (int k = 0; k < kClasses; ++k) {
        nd += tot[k];
        nm += tot[kClasses + k];
      }
      const int pd = tot[kCntPartDec], pm = tot[kCntPartMma];
      const bool fits = nd <= p.dec_cap && nm <= p.mma_cap && tot[kCntMerge] <= p.merge_cap &&
                        (int64_t)pd + pm <= p.part_cap;
      sh_state = fits ? 1 : 0;
      // Once: if the decode items are mostly full chunks (long sequences
      // split) and leave a last wave less than half full, grow the chunk so
      // that the count drops to whole waves.  Items of mixed sizes are left
      // to the largest-first order.
      const int P = max(1, p.dec_ctas), extra = nd % P;
      if (fits && iter == 0 && nd > P && extra > 0 && 2 * extra <= P && 4 * tot[0] >= 3 * nd) {
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
    }
    __syncthreads();
    if (sh_state) break;
  }
  if (sh_state == 2) {  // cannot happen with capacities from workspace_layout; emit nothing
    if (tid == 0) {
      p.header->n_dec = 0;
      p.header->n_mma = 0;
      p.header->n_merge = 0;
    }
    return;
  }

  // ---- emit: class k's items start after all larger classes' (largest first)
  const int cd = sh_chunk[0], cm = sh_chunk[1];
  {
    int base_dec = 0, base_mma = 0;
#pragma unroll
    for (int k = 0; k < kClasses; ++k) {
      s_cnt[k][tid] = base_dec + cnt[k];
      base_dec += tot[k];
      s_cnt[kClasses + k][tid] = base_mma + cnt[kClasses + k];
      base_mma += tot[kClasses + k];
    }
  }
  int off_grp = cnt[kCntMerge];
  int off_part = cnt[kCntPartDec] + cnt[kCntPartMma];
  {
    UnitIter t{i0, i1, U, B, 0, 0, 0, {}};
    for (iter_seek(t, p, seq_off); t.i < t.end; iter_next(t, p, seq_off)) {
      const SeqDesc& d = t.d;
      const int s = t.s, kvh = t.kvh, u = t.u;
      WorkItem* items = d.mma ? p.mma_items : p.dec_items;
      const int chunk = d.mma ? cm : cd;
      const int cbase = d.mma ? kClasses : 0;
      const int keys = unit_keys(d, u, p.G, p.causal);
      const int r0 = u * d.unit_rows;
      const int nr = min(d.rows - r0, d.unit_rows);
      int ns, per;
      split_of(keys, chunk, d.mma ? kMmaTileKeys : p.dec_tile_keys, ns, per);
      int grp = -1, part_base = 0;
      if (ns > 1) {
        grp = off_grp++;
        part_base = off_part;
        off_part += ns * nr;
        MergeGroup g;
        g.seq = s;
        g.kvh = kvh;
        g.row0 = r0;
        g.nrows = nr;
        g.nsplit = ns;
        g.part_base = part_base;
        g.pad0 = g.pad1 = 0;
        p.merges[grp] = g;
        p.tickets[grp] = 0;
      }
      const int full_cls = cbase + size_class(per, chunk);
      const int last_cls = cbase + size_class(keys - (ns - 1) * per, chunk);
      for (int sp = 0; sp < ns; ++sp) {
        WorkItem it;
        it.seq = s;
        it.kvh = kvh;
        it.row0 = r0;
        it.nrows = nr;
        it.kb = sp * per;
        it.ke = min(keys, (sp + 1) * per);
        it.part = ns > 1 ? part_base + sp * nr : -1;
        it.grp = grp;
        items[s_cnt[sp == ns - 1 ? last_cls : full_cls][tid]++] = it;
      }
    }
  }
  if (tid == 0) {
    int nd = 0, nm = 0;
#pragma unroll
    for (int k = 0; k < kClasses; ++k) {
      nd += tot[k];
      nm += tot[kClasses + k];
    }
    p.header->n_dec = nd;
    p.header->n_mma = nm;
    p.header->n_merge = tot[kCntMerge];
    p.header->chunk_dec = cd;
    p.header->chunk_mma = cm;
    p.header->part_rows = tot[kCntPartDec] + tot[kCntPartMma];
    p.header->dec_counter = 0;
    p.header->mma_counter = 0;
    p.header->merge_counter = 0;
  }
}

}  // namespace

cudaError_t launch_planner(const PlanParams& p, cudaStream_t s) {
  const size_t smem = (size_t)(p.B + 1) * sizeof(int);
  if (p.B > kMaxPlanSeqs) return cudaErrorInvalidValue;
  static unsigned long long done_mask = 0;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!(__atomic_load_n(&done_mask, __ATOMIC_ACQUIRE) & (1ull << dev))) {
    e = cudaFuncSetAttribute(plan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)((kMaxPlanSeqs + 1) * sizeof(int)));
    if (e != cudaSuccess) return e;
    __atomic_fetch_or(&done_mask, 1ull << dev, __ATOMIC_RELEASE);
  }
  e = launch_pdl(plan_kernel, dim3(1), dim3(kThreads), smem, s, p);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace pkv
