// Host/device shared declarations: the work plan written to the workspace by
// the planner kernel and read by the attention kernels, and the launch
// functions each translation unit exports to the host API.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <utility>

namespace pkv {

// Rows of one kv head of one sequence are (query token i, head-in-group g)
// pairs, row = i * G + g.
constexpr int kDecRows = 4;      // rows per CUDA-core work item
constexpr int kTcDecRows = 16;   // rows per tensor-core decode item (the MMA's N)
constexpr int kDecTileKeys = 64;  // keys per CUDA-core pipeline stage
constexpr int kMmaRows = 128;     // rows per tensor-core work item (M of the MMA)
constexpr int kMmaTileKeys = 128;  // keys per tensor-core pipeline stage
constexpr int kMaxSplits = 64;
constexpr int kMaxPlanSeqs = 32768;  // sequences per call (the planner keeps per-sequence offsets on chip)
// Shared prefixes ("cascade"): consecutive decode-shaped sequences whose
// block tables start with the same physical blocks form a group when there
// are at least kMinGroupSeqs of them; the group's common prefix (whole tiles
// of kMmaTileKeys keys visible to all its queries, at most kMaxPreTiles) is
// read once for all the group's rows, as multi-row tensor-core work.
constexpr int kMinGroupSeqs = 4;
constexpr int kMaxPreTiles = 31;

struct alignas(16) PlanHeader {
  int n_dec;        // CUDA-core work items
  int n_mma;        // tensor-core work items
  int n_merge;      // merge groups
  int chunk_dec;    // keys per split (CUDA-core path)
  int chunk_mma;    // keys per split (tensor-core path)
  int part_rows;    // partial rows used
  int dec_counter;  // work counters (dynamic item fetch), zeroed by the planner
  int mma_counter;
  int merge_counter;
  int n_pre;        // of the tensor-core items, those over shared prefixes (the last n_pre)
  int n_groups;     // prefix groups read once
  int mma_ctas;     // CTAs of the tensor-core kernel that take items (the rest leave their SMs to decode)
  int pad[4];
};

// One unit of attention work: `nrows` rows of sequence `seq`, kv head `kvh`,
// starting at row `row0`, over keys [kb, ke).  part < 0: normalise and write
// the output rows; otherwise write partial (m, l, acc) rows part .. part+nrows-1
// of merge group `grp`, and merge the group if this item finishes it last.
struct alignas(16) WorkItem {
  int seq, kvh, row0, nrows;
  int kb, ke, part, grp;
};

// Split-KV merge: rows row0 .. row0+nrows-1 of (seq, kvh) have nsplit
// partial states at part_base + p * nrows + r, and pre_n more (over a shared
// prefix, written before the split items run) at pre_base + c * pre_stride + r.
struct alignas(16) MergeGroup {
  int seq, kvh, row0, nrows;
  int nsplit, part_base, pre_base, pre_n;
  int pre_stride, pad0, pad1, pad2;
};

// A run of consecutive sequences s0 .. s1 sharing their first pre_keys keys
// (planner scratch).  Its rows (tokens query_start_loc[s0] ..
// query_start_loc[s1 + 1] - 1, G heads each) are cut into 128-row tiles; each
// (kv head, tile) reads the prefix in npre chunks, whose partial rows sit at
// part_off + (kvh * npre + c) * rows + row.
struct alignas(16) PreGroup {
  int s0, s1, pre_tiles, npre;
  int rows, item_off, part_off, valid;
};

struct WorkspaceLayout {
  size_t header_off, dec_off, mma_off, merge_off, ticket_off, seq_off, pre_off, ml_off, acc_off, total;
  int dec_cap, mma_cap, merge_cap, part_cap;
};

// Capacity arithmetic shared by the size queries and the forward call.
WorkspaceLayout workspace_layout(int B, int64_t T, int Hq, int Hkv, int D, size_t bytes_available,
                                 int num_sms, bool want_default_parts);

struct PlanParams {
  const int32_t* context_lens;
  const int32_t* query_start_loc;
  int B;
  int64_t T;
  int G;            // q heads per kv head
  int Hkv;
  int bs;
  int max_blocks;   // block table row length
  int causal;
  int mma_ok;       // tensor-core path available for this call
  int cascade;      // look for groups of sequences sharing a prefix (tensor-core decode only)
  const int32_t* block_tables;
  int dec_rows_max;  // rows <= this go to the decode-shaped path when mma_ok
  int dec_unit_rows;  // rows per decode-shaped item (4 CUDA-core, 16 tensor-core)
  int mma_unit_rows;  // rows per tensor-core item: the whole tokens that fit 128 rows, floor(128 / G) * G
  int dec_tile_keys;  // key tile of the decode-shaped kernel (splits are multiples)
  int target_dec, target_mma;  // desired item counts
  int dec_ctas;     // CTAs of the decode-shaped kernel (one wave of items)
  int sms;          // SMs of the device (CTAs of the tensor-core kernel)
  int side_by_side;  // the decode kernel may run beside the tensor-core kernel (no prefix items)
  int kv_key_bytes;  // K+V bytes per key of one kv head (2 * head_dim * element size)
  int min_chunk_dec, min_chunk_mma;
  int dec_cap, mma_cap, merge_cap, part_cap;
  PlanHeader* header;
  WorkItem* dec_items;
  WorkItem* mma_items;
  MergeGroup* merges;
  int* tickets;     // one per merge group, zeroed
  int* seq_pre;     // [B] scratch: keys of each sequence's prefix read by its group (0: none)
  int* seq_grp;     // [B] scratch: prefix group of each sequence
  uint32_t* seq_mask;  // [B] scratch: tiles equal to the previous sequence's
  int* seq_tmp;     // [B] scratch
  PreGroup* pre_groups;  // [B] scratch
  void* out;        // rows of invalid sequences are zeroed
  int out_row_bytes;  // bytes of one token's output row (Hq * D * elem)
  int* err;
  // The step's new K/V rows, written by CTAs 1 .. write_ctas of the
  // planner's grid (write_ctas 0: none).  write_mode 1: row copy of w_row
  // 16-byte chunks, strides in bytes; 2 / 3: FP8 quantizing write of bf16 /
  // fp32 rows of w_row elements, strides in elements.
  int write_ctas, write_mode, w_row;
  const void* wk;
  const void* wv;
  const int64_t* wslots;
  void* wkc;
  void* wvc;
  int64_t wT, w_num_slots, wk_stride, wv_stride;
  float wk_scale, wv_scale;
};

struct AttnParams {
  const void* q;
  void* out;
  const int32_t* block_tables;
  const int32_t* context_lens;
  const int32_t* query_start_loc;
  const PlanHeader* header;
  int* counter;
  const WorkItem* items;
  float2* part_ml;   // (m, l) per partial row, m in log2 units
  float* part_acc;   // [part_rows][D]
  const MergeGroup* groups;
  int* tickets;      // arrivals per merge group
  int Hq, Hkv, G, D, bs, max_blocks;
  int64_t num_blocks;
  float scale_log2;  // scale * log2(e) (times the K scale for an FP8 cache)
  float v_scale;     // output factor: the V scale for an FP8 cache, else 1
  int causal;
  int out_al32;      // out is 32-byte aligned (256-bit stores)
  int mma_unit_rows;  // rows of a full tensor-core item: floor(128 / G) * G (whole tokens)
  // The decode kernel launches beside the tensor-core kernel, after every
  // CTA of that kernel has seen the plan complete (they signal dependents
  // only then): it skips the grid-dependency wait, which would also wait for
  // the tensor-core kernel, and reads the plan from L2.
  int no_wait;
  int* err;
  // Bounded waits give up after wait_ns nanoseconds (0: the default, 2 s).
  uint64_t wait_ns;
  // Testing only (0 in every ordinary call): fault_tile >= 1 makes CTA 0's
  // K/V producer skip the loads and the arrival of its fault_tile-th key tile
  // (counting from 1), so that the waits for that tile run out and the
  // kernel's timeout path is exercised without any other fault.
  int fault_tile;
};

// Launch with programmatic stream serialization (the kernel may start before
// its predecessor in the stream finishes; it calls pdl_wait() before
// touching what the predecessor produces).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                              Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// launchers (return cudaGetLastError after the launch)
cudaError_t launch_kv_write(const void* k, const void* v, const int64_t* slots, void* kc, void* vc,
                            int64_t T, int64_t num_slots, int row_elems, int elem_bytes,
                            int64_t k_stride, int64_t v_stride, int* err, cudaStream_t s);
// FP8 (E4M3) cache: the quantising write (rows of bf16 or fp32, es bytes per
// element) and the CUDA-core decode kernel for bf16 q with head_dim 128
cudaError_t launch_kv_write_fp8(const void* k, const void* v, const int64_t* slots, void* kc, void* vc, int64_t T,
                                int64_t num_slots, int row_elems, int es, int64_t k_stride, int64_t v_stride,
                                float k_scale, float v_scale, int* err, cudaStream_t s);
cudaError_t launch_decode_fp8(const AttnParams& p, const CUtensorMap& kmap, const CUtensorMap& vmap, int grid,
                              cudaStream_t s);
cudaError_t decode_fp8_ctas_per_sm(int* ctas);
cudaError_t launch_planner(const PlanParams& p, cudaStream_t s);
// shared-prefix search for the planner (before it, on the same stream)
cudaError_t launch_prefix_search(const PlanParams& p, cudaStream_t s);
cudaError_t launch_decode(const AttnParams& p, const CUtensorMap& kmap, const CUtensorMap& vmap,
                          bool bf16, int grid, cudaStream_t s);
cudaError_t launch_mma(const AttnParams& p, const CUtensorMap& qmap, const CUtensorMap& kmap,
                       const CUtensorMap& vmap, const CUtensorMap& omap, int grid, cudaStream_t s);
// rows: the largest item row count (4, 8 or 16 rows of softmax per key)
cudaError_t launch_dectc(const AttnParams& p, int rows, const CUtensorMap& qmap, const CUtensorMap& kmap,
                         const CUtensorMap& vmap, int grid, cudaStream_t s);
// The same kernel over FP8 pools (rows <= 8): staged E4M3 tiles converted to
// fp16, fp16 MMAs; kmap / vmap are uint8 maps with {128, 1, bs, 1} boxes
cudaError_t launch_dectc_fp8(const AttnParams& p, int rows, const CUtensorMap& qmap, const CUtensorMap& kmap,
                             const CUtensorMap& vmap, int grid, cudaStream_t s);

// Sets the thread-local message pkv_last_error returns.
void set_last_error(const char* msg);

// Shared-memory bytes of the CUDA-core kernel, and its resident CTAs per SM
// (also sets the kernel's shared-memory opt-in on the current device).
int decode_smem_bytes(int D, int elem_bytes);
cudaError_t decode_ctas_per_sm(bool bf16, int D, int* ctas);

}  // namespace pkv
