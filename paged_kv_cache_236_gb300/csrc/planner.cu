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
// the GPU).  Splits write partial (max, sum, unnormalised accumulator) rows
// that the merge kernel combines.  The partial-row capacity is the
// workspace's; if a plan would not fit, chunks grow until it does.
//
// One CTA of 1024 threads; each thread owns a contiguous range of sequences
// so that block-wide exclusive scans give every item a fixed slot.
#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace {

constexpr int kThreads = 1024;

struct SeqDesc {
  int n, L, qstart;
  bool valid, mma;
  int rows, unit_rows, units;
};

__device__ __forceinline__ SeqDesc describe(const PlanParams& p, int s) {
  SeqDesc d;
  const int a = p.query_start_loc[s], b = p.query_start_loc[s + 1];
  d.L = p.context_lens[s];
  d.n = b - a;
  d.qstart = a;
  d.valid = a >= 0 && b >= a && (int64_t)b <= p.T && d.n <= d.L && d.L >= 0 &&
            (int64_t)d.L <= (int64_t)p.max_blocks * p.bs;
  d.rows = d.valid ? d.n * p.G : 0;
  d.mma = p.mma_ok && d.rows > p.dec_rows_max;
  d.unit_rows = d.mma ? kMmaRows : kDecRows;
  d.units = (d.rows + d.unit_rows - 1) / d.unit_rows;
  return d;
}

// Keys a unit must visit: rows [r0, r1) of the sequence.
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

struct Counts {
  long long dec_items, mma_items, merges, part_rows;
};

__device__ __forceinline__ Counts count_seq(const PlanParams& p, const SeqDesc& d, int chunk_dec,
                                            int chunk_mma) {
  Counts c = {0, 0, 0, 0};
  for (int u = 0; u < d.units; ++u) {
    const int keys = unit_keys(d, u, p.G, p.causal);
    const int nr = min(d.rows - u * d.unit_rows, d.unit_rows);
    int ns, per;
    split_of(keys, d.mma ? chunk_mma : chunk_dec, d.mma ? kMmaTileKeys : kDecTileKeys, ns, per);
    if (d.mma)
      c.mma_items += ns;
    else
      c.dec_items += ns;
    if (ns > 1) {
      c.merges += 1;
      c.part_rows += (long long)ns * nr;
    }
  }
  c.dec_items *= p.Hkv;
  c.mma_items *= p.Hkv;
  c.merges *= p.Hkv;
  c.part_rows *= p.Hkv;
  return c;
}

// Block-wide exclusive scan of four 64-bit counters; returns this thread's
// offsets and (via `total`) the sums.
__device__ void block_scan4(const long long v[4], long long off[4], long long total[4]) {
  __shared__ long long warp_sums[kThreads / 32][4];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  long long incl[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    long long x = v[k];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const long long y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    incl[k] = x;
    if (lane == 31) warp_sums[warp][k] = x;
  }
  __syncthreads();
  if (warp == 0) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      long long x = warp_sums[lane][k];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const long long y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
      }
      warp_sums[lane][k] = x;  // inclusive over warps
    }
  }
  __syncthreads();
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const long long before = warp > 0 ? warp_sums[warp - 1][k] : 0;
    off[k] = before + incl[k] - v[k];
    total[k] = warp_sums[kThreads / 32 - 1][k];
  }
  __syncthreads();
}

__global__ void __launch_bounds__(kThreads) plan_kernel(PlanParams p) {
  const int tid = threadIdx.x;
  const int per_thread = (p.B + kThreads - 1) / kThreads;
  const int s0 = min(p.B, tid * per_thread);
  const int s1 = min(p.B, s0 + per_thread);

  // --- total work per path (keys x kv heads) and invalid-sequence cleanup ---
  long long w[4] = {0, 0, 0, 0};
  for (int s = s0; s < s1; ++s) {
    const SeqDesc d = describe(p, s);
    if (!d.valid) {
      raise_error(p.err, PKV_DEVERR_BAD_SEQUENCE);
      const int a = p.query_start_loc[s], b = p.query_start_loc[s + 1];
      if (a >= 0 && b > a && (int64_t)b <= p.T) {  // zero the rows that are addressable
        int4* o = reinterpret_cast<int4*>(static_cast<uint8_t*>(p.out) + (int64_t)a * p.out_row_bytes);
        const int64_t n16 = (int64_t)(b - a) * p.out_row_bytes / 16;
        for (int64_t i = 0; i < n16; ++i) o[i] = make_int4(0, 0, 0, 0);
      }
      continue;
    }
    for (int u = 0; u < d.units; ++u) w[d.mma ? 1 : 0] += (long long)unit_keys(d, u, p.G, p.causal) * p.Hkv;
  }
  long long woff[4], wtot[4];
  block_scan4(w, woff, wtot);

  __shared__ int sh_chunk[2];
  __shared__ int sh_done;
  if (tid == 0) {
    long long cd = (wtot[0] + p.target_dec - 1) / max(1, p.target_dec);
    long long cm = (wtot[1] + p.target_mma - 1) / max(1, p.target_mma);
    cd = max(cd, (long long)p.min_chunk_dec);
    cm = max(cm, (long long)p.min_chunk_mma);
    cd = (cd + kDecTileKeys - 1) / kDecTileKeys * kDecTileKeys;
    cm = (cm + kMmaTileKeys - 1) / kMmaTileKeys * kMmaTileKeys;
    sh_chunk[0] = (int)min(cd, (long long)(1 << 30));
    sh_chunk[1] = (int)min(cm, (long long)(1 << 30));
  }
  __syncthreads();

  // --- grow chunks until the plan fits the workspace ---
  long long c[4], off[4], tot[4];
  for (int iter = 0;; ++iter) {
    const int cd = sh_chunk[0], cm = sh_chunk[1];
    c[0] = c[1] = c[2] = c[3] = 0;
    long long part_dec = 0, part_mma = 0;
    for (int s = s0; s < s1; ++s) {
      const SeqDesc d = describe(p, s);
      if (!d.valid || d.rows == 0) continue;
      const Counts k = count_seq(p, d, cd, cm);
      c[0] += k.dec_items;
      c[1] += k.mma_items;
      c[2] += k.merges;
      c[3] += k.part_rows;
      (d.mma ? part_mma : part_dec) += k.part_rows;
    }
    block_scan4(c, off, tot);
    long long pd[4] = {part_dec, part_mma, 0, 0}, pdo[4], pdt[4];
    block_scan4(pd, pdo, pdt);
    if (tid == 0) {
      const bool fits = tot[0] <= p.dec_cap && tot[1] <= p.mma_cap && tot[2] <= p.merge_cap &&
                        tot[3] <= p.part_cap;
      sh_done = fits ? 1 : 0;
      if (!fits) {
        if (iter >= 40) {
          raise_error(p.err, PKV_DEVERR_PLAN_OVERFLOW);
          sh_done = 2;
        }
        const bool dec_over = tot[0] > p.dec_cap || pdt[0] >= pdt[1];
        const bool mma_over = tot[1] > p.mma_cap || pdt[1] > pdt[0];
        if (dec_over) sh_chunk[0] = (int)min(2LL * cd, (long long)(1 << 30));
        if (mma_over) sh_chunk[1] = (int)min(2LL * cm, (long long)(1 << 30));
      }
    }
    __syncthreads();
    if (sh_done) break;
  }
  if (sh_done == 2) {  // cannot happen with capacities from workspace_layout; emit nothing
    if (tid == 0) {
      p.header->n_dec = 0;
      p.header->n_mma = 0;
      p.header->n_merge = 0;
    }
    return;
  }

  // --- emit ---
  const int cd = sh_chunk[0], cm = sh_chunk[1];
  long long o_dec = off[0], o_mma = off[1], o_mrg = off[2], o_part = off[3];
  for (int s = s0; s < s1; ++s) {
    const SeqDesc d = describe(p, s);
    if (!d.valid || d.rows == 0) continue;
    WorkItem* items = d.mma ? p.mma_items : p.dec_items;
    long long& o_it = d.mma ? o_mma : o_dec;
    for (int kvh = 0; kvh < p.Hkv; ++kvh) {
      for (int u = 0; u < d.units; ++u) {
        const int keys = unit_keys(d, u, p.G, p.causal);
        const int r0 = u * d.unit_rows;
        const int nr = min(d.rows - r0, d.unit_rows);
        int ns, per;
        split_of(keys, d.mma ? cm : cd, d.mma ? kMmaTileKeys : kDecTileKeys, ns, per);
        if (ns > 1) {
          MergeGroup g;
          g.seq = s;
          g.kvh = kvh;
          g.row0 = r0;
          g.nrows = nr;
          g.nsplit = ns;
          g.part_base = (int)o_part;
          g.pad0 = g.pad1 = 0;
          p.merges[o_mrg++] = g;
        }
        for (int sp = 0; sp < ns; ++sp) {
          WorkItem it;
          it.seq = s;
          it.kvh = kvh;
          it.row0 = r0;
          it.nrows = nr;
          it.kb = sp * per;
          it.ke = min(keys, (sp + 1) * per);
          it.part = ns > 1 ? (int)(o_part + (long long)sp * nr) : -1;
          it.pad = 0;
          items[o_it++] = it;
        }
        if (ns > 1) o_part += (long long)ns * nr;
      }
    }
  }
  if (tid == 0) {
    p.header->n_dec = (int)tot[0];
    p.header->n_mma = (int)tot[1];
    p.header->n_merge = (int)tot[2];
    p.header->chunk_dec = cd;
    p.header->chunk_mma = cm;
    p.header->part_rows = (int)tot[3];
    p.header->dec_counter = 0;
    p.header->mma_counter = 0;
    p.header->merge_counter = 0;
  }
}

}  // namespace

cudaError_t launch_planner(const PlanParams& p, cudaStream_t s) {
  plan_kernel<<<1, kThreads, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace pkv
