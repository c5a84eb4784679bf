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
// One CTA of kThreads threads; each thread owns a contiguous range of
// (sequence, kv head) pairs, and block-wide exclusive scans give every item
// a fixed slot (items ordered by size class, then pair, then row unit and
// split).
#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kClasses = 8;            // item size classes
constexpr int kNumCounts = 2 * kClasses + 2;  // dec classes, mma classes, merges, partial rows

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

// Block-wide exclusive scan of K ints per thread (in place); totals[] gets the sums.
template <int K>
__device__ void block_scan(int (&v)[K], int (&totals)[K]) {
  __shared__ int warp_tot[kWarps][K];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl[K];
#pragma unroll
  for (int k = 0; k < K; ++k) {
    int x = v[k];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    incl[k] = x;
    if (lane == 31) warp_tot[warp][k] = x;
  }
  __syncthreads();
#pragma unroll
  for (int k = 0; k < K; ++k) {
    int before = 0, tot = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const int t = warp_tot[w][k];
      before += w < warp ? t : 0;
      tot += t;
    }
    v[k] = before + incl[k] - v[k];
    totals[k] = tot;
  }
  __syncthreads();
}

__global__ void __launch_bounds__(kThreads) plan_kernel(PlanParams p) {
  // The attention kernel may start its prologue while this plans (it waits
  // for this grid).  This grid waits for its own predecessor before reading
  // the metadata, which that predecessor may have produced.
  pdl_launch_dependents();
  pdl_wait();
  const int tid = threadIdx.x;
  const int np = p.B * p.Hkv;  // (sequence, kv head) pairs
  const int per_thread = (np + kThreads - 1) / kThreads;
  const int q0 = min(np, tid * per_thread);
  const int q1 = min(np, q0 + per_thread);

  // ---- total work per path (keys of all units of all pairs); zero the rows of invalid sequences
  __shared__ unsigned long long sh_work[2];
  __shared__ int sh_chunk[2];
  __shared__ int sh_state;
  if (tid < 2) sh_work[tid] = 0;
  __syncthreads();
  unsigned long long w_dec = 0, w_mma = 0;
  for (int q = q0; q < q1; ++q) {
    const int s = q / p.Hkv;
    const SeqDesc d = describe(p, s);
    if (!d.valid) {
      if (q % p.Hkv == 0) {  // once per sequence
        raise_error(p.err, PKV_DEVERR_BAD_SEQUENCE);
        const int a = p.query_start_loc[s], b = p.query_start_loc[s + 1];
        if (a >= 0 && b > a && (int64_t)b <= p.T) {  // zero the rows that are addressable
          int4* o = reinterpret_cast<int4*>(static_cast<uint8_t*>(p.out) + (int64_t)a * p.out_row_bytes);
          const int64_t n16 = (int64_t)(b - a) * p.out_row_bytes / 16;
          for (int64_t i = 0; i < n16; ++i) o[i] = make_int4(0, 0, 0, 0);
        }
      }
      continue;
    }
    unsigned long long w = 0;
    for (int u = 0; u < d.units; ++u) w += (unsigned long long)unit_keys(d, u, p.G, p.causal);
    (d.mma ? w_mma : w_dec) += w;
  }
  // warp sums, then one thread adds the warps' (no contended 64-bit atomics)
  __shared__ unsigned long long sh_wsum[kWarps][2];
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
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      sh_work[0] += sh_wsum[w][0];
      sh_work[1] += sh_wsum[w][1];
    }
    unsigned long long cd = (sh_work[0] + p.target_dec - 1) / (unsigned long long)max(1, p.target_dec);
    unsigned long long cm = (sh_work[1] + p.target_mma - 1) / (unsigned long long)max(1, p.target_mma);
    cd = max(cd, (unsigned long long)p.min_chunk_dec);
    cm = max(cm, (unsigned long long)p.min_chunk_mma);
    cd = (cd + p.dec_tile_keys - 1) / p.dec_tile_keys * p.dec_tile_keys;
    cm = (cm + kMmaTileKeys - 1) / kMmaTileKeys * kMmaTileKeys;
    sh_chunk[0] = (int)min(cd, (unsigned long long)(1 << 30));
    sh_chunk[1] = (int)min(cm, (unsigned long long)(1 << 30));
  }
  __syncthreads();

  // ---- grow chunks until the plan fits the workspace
  for (int iter = 0;; ++iter) {
    const int cd = sh_chunk[0], cm = sh_chunk[1];
    int c[5] = {0, 0, 0, 0, 0};  // dec items, mma items, merges, partial rows (dec), partial rows (mma)
    for (int q = q0; q < q1; ++q) {
      const SeqDesc d = describe(p, q / p.Hkv);
      if (!d.valid || d.rows == 0) continue;
      for (int u = 0; u < d.units; ++u) {
        int ns, per;
        split_of(unit_keys(d, u, p.G, p.causal), d.mma ? cm : cd, d.mma ? kMmaTileKeys : p.dec_tile_keys, ns, per);
        c[d.mma ? 1 : 0] += ns;
        if (ns > 1) {
          c[2] += 1;
          c[d.mma ? 4 : 3] += ns * min(d.rows - u * d.unit_rows, d.unit_rows);
        }
      }
    }
    int tot[5];
    block_scan<5>(c, tot);
    if (tid == 0) {
      const bool fits = tot[0] <= p.dec_cap && tot[1] <= p.mma_cap && tot[2] <= p.merge_cap &&
                        (int64_t)tot[3] + tot[4] <= p.part_cap;
      sh_state = fits ? 1 : 0;
      if (!fits) {
        if (iter >= 40) {
          raise_error(p.err, PKV_DEVERR_PLAN_OVERFLOW);
          sh_state = 2;
        }
        const bool dec_over = tot[0] > p.dec_cap || tot[3] >= tot[4];
        const bool mma_over = tot[1] > p.mma_cap || tot[4] > tot[3];
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

  // ---- count items per size class, scan, emit largest class first
  const int cd = sh_chunk[0], cm = sh_chunk[1];
  __shared__ int s_ctr[kNumCounts][kThreads];  // per-thread counters, then running offsets
#pragma unroll
  for (int k = 0; k < kNumCounts; ++k) s_ctr[k][tid] = 0;
  for (int q = q0; q < q1; ++q) {
    const SeqDesc d = describe(p, q / p.Hkv);
    if (!d.valid || d.rows == 0) continue;
    const int chunk = d.mma ? cm : cd;
    const int cb = d.mma ? kClasses : 0;
    for (int u = 0; u < d.units; ++u) {
      const int keys = unit_keys(d, u, p.G, p.causal);
      int ns, per;
      split_of(keys, chunk, d.mma ? kMmaTileKeys : p.dec_tile_keys, ns, per);
      s_ctr[cb + size_class(per, chunk)][tid] += ns - 1;  // all splits but the last are full
      s_ctr[cb + size_class(keys - (ns - 1) * per, chunk)][tid] += 1;
      if (ns > 1) {
        s_ctr[2 * kClasses][tid] += 1;
        s_ctr[2 * kClasses + 1][tid] += ns * min(d.rows - u * d.unit_rows, d.unit_rows);
      }
    }
  }
  int cnt[kNumCounts];
#pragma unroll
  for (int k = 0; k < kNumCounts; ++k) cnt[k] = s_ctr[k][tid];
  int tot[kNumCounts];
  block_scan<kNumCounts>(cnt, tot);
  {
    int base_dec = 0, base_mma = 0;
#pragma unroll
    for (int k = 0; k < kClasses; ++k) {
      s_ctr[k][tid] = base_dec + cnt[k];
      base_dec += tot[k];
      s_ctr[kClasses + k][tid] = base_mma + cnt[kClasses + k];
      base_mma += tot[kClasses + k];
    }
    s_ctr[2 * kClasses][tid] = cnt[2 * kClasses];
    s_ctr[2 * kClasses + 1][tid] = cnt[2 * kClasses + 1];
  }
  int* off_grp = &s_ctr[2 * kClasses][tid];
  int* off_part = &s_ctr[2 * kClasses + 1][tid];
  for (int q = q0; q < q1; ++q) {
    const int s = q / p.Hkv, kvh = q - s * p.Hkv;
    const SeqDesc d = describe(p, s);
    if (!d.valid || d.rows == 0) continue;
    WorkItem* items = d.mma ? p.mma_items : p.dec_items;
    const int chunk = d.mma ? cm : cd;
    const int cbase = d.mma ? kClasses : 0;
    for (int u = 0; u < d.units; ++u) {
      const int keys = unit_keys(d, u, p.G, p.causal);
      const int r0 = u * d.unit_rows;
      const int nr = min(d.rows - r0, d.unit_rows);
      int ns, per;
      split_of(keys, chunk, d.mma ? kMmaTileKeys : p.dec_tile_keys, ns, per);
      int grp = -1, part_base = 0;
      if (ns > 1) {
        grp = (*off_grp)++;
        part_base = *off_part;
        *off_part += ns * nr;
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
        items[s_ctr[sp == ns - 1 ? last_cls : full_cls][tid]++] = it;
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
    p.header->n_merge = tot[2 * kClasses];
    p.header->chunk_dec = cd;
    p.header->chunk_mma = cm;
    p.header->part_rows = tot[2 * kClasses + 1];
    p.header->dec_counter = 0;
    p.header->mma_counter = 0;
    p.header->merge_counter = 0;
  }
}

}  // namespace

cudaError_t launch_planner(const PlanParams& p, cudaStream_t s) {
  const cudaError_t e = launch_pdl(plan_kernel, dim3(1), dim3(kThreads), 0, s, p);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace pkv
