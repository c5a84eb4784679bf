/*
 * paged_kv.h - C ABI of a GB300 (sm_103a) library for attention over a
 * block-paged KV cache.
 *
 * The operations follow the source pages:
 *   - "ADR 004: Paged Attention Serving Integration" (Decision 4): the model
 *     writes each layer's K/V rows into a block allocator and reads them back
 *     through paged_attention_forward; prefill chunks and decode steps share
 *     one call (Consequences).
 *   - "Paged Attention 基础 - 原理与实现进度", section 2: a sequence's
 *     logical positions map to physical blocks through a block table; a
 *     query gathers its keys block by block, applies the causal mask and
 *     computes softmax(QK^T)V; several tables may name the same physical
 *     block (prefix sharing).  Section 3.2 names the metadata: block_tables,
 *     slot_mapping, context_lens.
 *   - Dao-AILab/flash-attention issue #660: several query tokens per
 *     sequence (speculative decoding) next to single-token decode; the caller
 *     owns the cache manager and calls kernels only.
 *
 * Layouts (row-major, innermost dimension contiguous):
 *   block pool, per layer   k_cache, v_cache  [num_blocks, block_size, num_kv_heads, head_dim]
 *   new K/V rows            k, v              [num_tokens, num_kv_heads, head_dim]
 *                                             (token stride may exceed num_kv_heads*head_dim)
 *   queries / output        q, out            [num_tokens, num_q_heads, head_dim]
 *   slot_mapping            int64  [num_tokens]; slot = block * block_size + offset; < 0 skips
 *   block_tables            int32  [num_seqs, max_blocks_per_seq]; entries past a sequence's
 *                                  last block are ignored (may be -1)
 *   context_lens            int32  [num_seqs]; tokens in the cache AFTER this step's write,
 *                                  the sequence's new (query) tokens included
 *   query_start_loc         int32  [num_seqs + 1]; query rows of sequence s are
 *                                  q[query_start_loc[s] : query_start_loc[s+1]]
 *
 * Semantics: query i of a sequence with n queries and L tokens sits at
 * position L - n + i; with causal != 0 it attends keys 0 .. L-n+i, otherwise
 * all L keys.  Query head h reads kv head h / (num_q_heads / num_kv_heads).
 * The result is softmax(scale * q k^T) v accumulated in fp32 and cast to the
 * dtype of q (round to nearest even).
 *
 * Ownership: every buffer is the caller's (device memory unless stated);
 * the library allocates no device memory and keeps no state across calls
 * except the cached driver entry point and the sticky device error word.
 * Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy default
 * stream).  Pointers must be 16-byte aligned.
 *
 * Errors: host-checkable problems return a status before any launch and set a
 * thread-local message (pkv_last_error).  Metadata that only the device sees
 * never faults; each case sets a bit in the sticky device error word that
 * pkv_device_errors reads:
 *   - a slot outside the pool: that token's write is skipped
 *     (PKV_DEVERR_SLOT_OUT_OF_RANGE);
 *   - a block id outside [0, num_blocks) among a sequence's first
 *     ceil(context_len / block_size) table entries: that block is read as a
 *     block of zeros, i.e. its keys score 0 and carry zero values, and the
 *     rest of the sequence is attended as usual
 *     (PKV_DEVERR_BLOCK_OUT_OF_RANGE);
 *   - a sequence with more queries than tokens, a non-monotone
 *     query_start_loc or a context longer than its table: the rows it
 *     addresses are written as zeros (PKV_DEVERR_BAD_SEQUENCE).
 */
#ifndef PAGED_KV_H_
#define PAGED_KV_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  PKV_OK = 0,
  PKV_ERR_INVALID_ARG = 1,  /* bad pointer, size, alignment or shape */
  PKV_ERR_UNSUPPORTED = 2,  /* valid but not implemented (dtype, head_dim, block_size, GPU) */
  PKV_ERR_CUDA = 3,         /* a CUDA runtime/driver call or a launch failed */
  PKV_ERR_WORKSPACE = 4,    /* workspace missing or smaller than required */
  PKV_ERR_OUT_OF_BLOCKS = 5 /* block manager: free and evictable blocks do not cover the request */
} pkv_status;

typedef enum {
  PKV_DTYPE_F32 = 0,
  PKV_DTYPE_BF16 = 1,
  PKV_DTYPE_FP8_E4M3 = 2  /* cache codes only: see paged_kv_write_fp8 */
} pkv_dtype;

/*
 * Host hints for paged_attention_forward (bit flags).
 *
 * PKV_HINT_SHARED_PREFIX: consecutive sequences of the batch may start with
 * the same physical blocks (prefix caching: several requests built on one
 * cached prompt; "PagedAttention" prefix sharing).  The call then looks for
 * runs of at least 4 decode-shaped sequences whose block tables agree on
 * their first whole 128-key tiles (up to 31 tiles, keys every query of the
 * run sees) and reads those keys once for the whole run, as tensor-core work
 * over all the run's query rows; each member's remaining keys are read as
 * usual and the two parts merged (the result is the same attention, up to
 * rounding).  Only on the bf16 / head_dim 128 tensor-core decode path;
 * ignored elsewhere.  Costs a short scan of the block tables per call.
 */
#define PKV_HINT_SHARED_PREFIX 0x1

/* Device error word bits (pkv_device_errors). */
#define PKV_DEVERR_SLOT_OUT_OF_RANGE 0x1   /* slot_mapping entry >= num_blocks * block_size */
#define PKV_DEVERR_BLOCK_OUT_OF_RANGE 0x2  /* block table entry outside [0, num_blocks) */
#define PKV_DEVERR_BAD_SEQUENCE 0x4        /* q_len < 0, q_len > context_len, context too long */
#define PKV_DEVERR_TIMEOUT 0x8             /* a bounded in-kernel wait gave up */
#define PKV_DEVERR_PLAN_OVERFLOW 0x10      /* work list did not fit the workspace */
#define PKV_DEVERR_INTERNAL 0x20           /* a kernel found its launch configuration unusable */

/*
 * paged_kv_write - scatter new K/V rows into the block pool.
 *
 * For every t < num_tokens with s = slot_mapping[t] >= 0:
 *   k_cache[s / block_size][s % block_size][:][:] = k[t][:][:]   (and v likewise)
 * A bit-exact copy in `dtype`.  ("ADR 004", Decision 4; "Paged Attention 基础",
 * section 2: token position -> physical block and slot.)
 *
 *   k, v            device, [num_tokens, num_kv_heads, head_dim], token stride
 *                   k_token_stride / v_token_stride ELEMENTS (>= num_kv_heads*head_dim;
 *                   0 means dense)
 *   slot_mapping    device int64 [num_tokens]
 *   k_cache,v_cache device [num_blocks, block_size, num_kv_heads, head_dim]
 * Two tokens with the same non-negative slot in one call: which one lands is
 * unspecified.  Writes into a block shared by several tables are the
 * caller's responsibility (copy-on-write belongs to the cache manager).
 * num_tokens == 0 is a no-op.
 */
pkv_status paged_kv_write(const void* k, const void* v, const int64_t* slot_mapping,
                          void* k_cache, void* v_cache,
                          int64_t num_tokens, int64_t num_blocks, int32_t block_size,
                          int32_t num_kv_heads, int32_t head_dim,
                          int64_t k_token_stride, int64_t v_token_stride,
                          pkv_dtype dtype, void* stream);

/*
 * paged_attention_workspace_size - bytes of device workspace that
 * paged_attention_forward wants for a batch of this shape (an upper bound
 * of what it uses; any smaller size >= paged_attention_workspace_min also
 * works, with fewer KV splits).  Pure host arithmetic.
 */
size_t paged_attention_workspace_size(int32_t num_seqs, int64_t num_tokens, int32_t num_q_heads,
                                      int32_t num_kv_heads, int32_t head_dim);

/* Smallest workspace paged_attention_forward accepts for this shape. */
size_t paged_attention_workspace_min(int32_t num_seqs, int64_t num_tokens, int32_t num_q_heads,
                                     int32_t num_kv_heads, int32_t head_dim);

/*
 * paged_attention_forward - varlen attention through per-sequence block
 * tables.  One call serves prefill chunks, single-token decode and
 * multi-token speculative verification ("ADR 004", Consequences;
 * flash-attention issue #660), with GQA/MQA (num_q_heads a multiple of
 * num_kv_heads) and physically shared blocks.
 *
 *   q               device [num_tokens, num_q_heads, head_dim], dtype
 *   k_cache,v_cache device [num_blocks, block_size, num_kv_heads, head_dim], dtype
 *   block_tables    device int32 [num_seqs, max_blocks_per_seq]
 *   context_lens    device int32 [num_seqs]
 *   query_start_loc device int32 [num_seqs + 1], query_start_loc[num_seqs] == num_tokens
 *   out             device [num_tokens, num_q_heads, head_dim], dtype; every row of
 *                   every sequence is written
 *   max_query_len   host hint: an upper bound of every sequence's query count, or
 *                   0 if unknown (used to pick the kernels; a smaller value still
 *                   gives the right rows, possibly slower)
 *   scale           logit scale (e.g. 1/sqrt(head_dim))
 *   causal          non-zero: bottom-right aligned causal mask
 *   hints           PKV_HINT_* bits (0: none)
 *   workspace       device scratch of workspace_bytes (>= paged_attention_workspace_min),
 *                   256-byte aligned; overwritten by the call; must not be shared by
 *                   calls that may run concurrently
 * Supported: dtype bf16 or f32; head_dim 64 or 128; block_size 8, 16, 32 or 64;
 * num_q_heads / num_kv_heads <= 128; num_seqs <= 32768 (PKV_ERR_UNSUPPORTED
 * beyond).
 * Invalid metadata is handled as the error notes at the top of this file
 * state (zero rows for an invalid sequence; an out-of-pool block id read as
 * a block of zeros).
 */
pkv_status paged_attention_forward(const void* q, const void* k_cache, const void* v_cache,
                                   const int32_t* block_tables, const int32_t* context_lens,
                                   const int32_t* query_start_loc, void* out,
                                   int32_t num_seqs, int64_t num_tokens, int32_t num_q_heads,
                                   int32_t num_kv_heads, int32_t head_dim, int64_t num_blocks,
                                   int32_t block_size, int32_t max_blocks_per_seq,
                                   int32_t max_query_len, float scale, int32_t causal,
                                   int32_t hints, void* workspace, size_t workspace_bytes,
                                   pkv_dtype dtype, void* stream);

/*
 * paged_kv_write_attention_forward - paged_kv_write of a step's new K/V rows
 * followed by paged_attention_forward over the pools, in one call and one
 * launch fewer ("ADR 004", Consequences: the model writes a layer's new K/V
 * and then attends, prefill and decode alike).  The results are those of the
 * two calls made in that order on `stream`.
 *
 *   k, v, slot_mapping, num_new_tokens, k_token_stride, v_token_stride
 *                   the new rows, as paged_kv_write takes them ([num_new_tokens,
 *                   num_kv_heads, head_dim] of `dtype`, strides in elements, 0
 *                   means dense; slots < 0 skipped)
 *   the rest        as paged_attention_forward
 * When every row start is 16-byte aligned, the rows are copied by extra CTAs
 * of the planner's launch (the attention kernels wait for that launch, so
 * they read the new rows); otherwise the write kernel runs first.  Errors as
 * for the two calls (the write's arguments are checked before any launch).
 */
pkv_status paged_kv_write_attention_forward(const void* k, const void* v, const int64_t* slot_mapping,
                                            int64_t num_new_tokens, int64_t k_token_stride,
                                            int64_t v_token_stride, const void* q, const void* k_cache,
                                            const void* v_cache, const int32_t* block_tables,
                                            const int32_t* context_lens, const int32_t* query_start_loc,
                                            void* out, int32_t num_seqs, int64_t num_tokens,
                                            int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                            int64_t num_blocks, int32_t block_size, int32_t max_blocks_per_seq,
                                            int32_t max_query_len, float scale, int32_t causal, int32_t hints,
                                            void* workspace, size_t workspace_bytes, pkv_dtype dtype,
                                            void* stream);

/*
 * paged_attention_forward_static_ws - paged_attention_forward for callers
 * that cannot allocate device memory (no counterpart on the source pages).
 *
 * Same arguments and results as paged_attention_forward, without the
 * workspace: the scratch is a static array compiled into the library
 * (paged_attention_static_workspace_bytes(), 8 MiB), present on every GPU that
 * loads the library until the process exits.  Meant for code that runs under
 * an allocator which forbids new device allocations once started, or that
 * can only pass through buffers someone else registered.  The call allocates
 * nothing (no cudaMalloc / cudaFree, no allocating library routine).
 *   - A batch whose paged_attention_workspace_min exceeds the static size is
 *     rejected with PKV_ERR_WORKSPACE before any launch.
 *   - Each call looks up the array's device address (cudaGetSymbolAddress,
 *     with the current device); the first lookup on a device may load the
 *     library's device code, so make the first call on each device before
 *     any stream capture.
 *   - Every call on a device uses the same array, which keeps the last call's
 *     contents (each call rewrites what it reads).  Calls whose GPU work can
 *     overlap (other streams, unordered host threads) race on it: serialise
 *     them.
 */
pkv_status paged_attention_forward_static_ws(const void* q, const void* k_cache, const void* v_cache,
                                             const int32_t* block_tables, const int32_t* context_lens,
                                             const int32_t* query_start_loc, void* out,
                                             int32_t num_seqs, int64_t num_tokens, int32_t num_q_heads,
                                             int32_t num_kv_heads, int32_t head_dim, int64_t num_blocks,
                                             int32_t block_size, int32_t max_blocks_per_seq,
                                             int32_t max_query_len, float scale, int32_t causal,
                                             int32_t hints, pkv_dtype dtype, void* stream);

/*
 * FP8 KV cache (the library's own format; the source pages name no cache
 * precision).  Each pool element is an 8-bit E4M3 code (OCP "e4m3fn": 1 sign,
 * 4 exponent bits with bias 7, 3 mantissa bits, largest finite value 448, no
 * infinities), with one fp32 scale for the K pool and one for the V pool,
 * chosen by the caller (e.g. per layer):
 *   code = E4M3(RNE(x / scale)), x / scale an IEEE fp32 division, magnitudes
 *          beyond 448 saturated to +-448
 *   value read = code * scale.
 * Pools are [num_blocks, block_size, num_kv_heads, head_dim] bytes: half the
 * bytes of bf16, so decode, which reads every cached row once per step,
 * moves half the memory.
 *
 * paged_kv_write_fp8 - paged_kv_write into FP8 pools: rows k, v of `dtype`
 * (bf16 or f32; token strides in elements, multiples of 16 bytes; 0 means
 * dense) are encoded with k_scale / v_scale and scattered by slot_mapping
 * (slots < 0 skipped).  num_kv_heads * head_dim must be a multiple of 16.
 */
pkv_status paged_kv_write_fp8(const void* k, const void* v, const int64_t* slot_mapping,
                              void* k_cache, void* v_cache,
                              int64_t num_tokens, int64_t num_blocks, int32_t block_size,
                              int32_t num_kv_heads, int32_t head_dim,
                              int64_t k_token_stride, int64_t v_token_stride,
                              pkv_dtype dtype, float k_scale, float v_scale, void* stream);

/*
 * paged_attention_forward_fp8kv - paged_attention_forward with FP8 pools:
 * q and out bf16, k_cache / v_cache E4M3 codes read as code * k_scale and
 * code * v_scale; the same metadata, workspace and results otherwise
 * (softmax(scale q k^T) v, fp32 accumulation).  head_dim 128 (other head
 * sizes: PKV_ERR_UNSUPPORTED); any block_size, GQA group and query count of
 * paged_attention_forward.  When max_query_len > 0, the group size
 * num_q_heads / num_kv_heads is a power of two and max_query_len times it is
 * at most 8, the tensor-core decode kernel runs: staged code tiles are
 * converted to fp16 in shared memory, q is rounded to fp16 (|q| must stay
 * below 65504) and the MMAs take fp16 operands.  Otherwise the CUDA-core
 * kernel runs, K and V converted to fp32 in registers.
 * PKV_HINT_SHARED_PREFIX is ignored.
 */
pkv_status paged_attention_forward_fp8kv(const void* q, const void* k_cache, const void* v_cache,
                                         const int32_t* block_tables, const int32_t* context_lens,
                                         const int32_t* query_start_loc, void* out,
                                         int32_t num_seqs, int64_t num_tokens, int32_t num_q_heads,
                                         int32_t num_kv_heads, int32_t head_dim, int64_t num_blocks,
                                         int32_t block_size, int32_t max_blocks_per_seq,
                                         int32_t max_query_len, float scale, int32_t causal,
                                         float k_scale, float v_scale, int32_t hints, void* workspace,
                                         size_t workspace_bytes, void* stream);

/*
 * paged_kv_write_attention_forward_fp8kv - paged_kv_write_fp8 of a step's new
 * rows (of row_dtype, bf16 or f32, 16-byte aligned with strides of multiples
 * of 16 bytes) followed by paged_attention_forward_fp8kv, in one call; the
 * rows are encoded by extra CTAs of the planner's launch.  Arguments and
 * errors as for the two calls.
 */
pkv_status paged_kv_write_attention_forward_fp8kv(
    const void* k, const void* v, const int64_t* slot_mapping, int64_t num_new_tokens, int64_t k_token_stride,
    int64_t v_token_stride, pkv_dtype row_dtype, const void* q, const void* k_cache, const void* v_cache,
    const int32_t* block_tables, const int32_t* context_lens, const int32_t* query_start_loc, void* out,
    int32_t num_seqs, int64_t num_tokens, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
    int64_t num_blocks, int32_t block_size, int32_t max_blocks_per_seq, int32_t max_query_len, float scale,
    int32_t causal, float k_scale, float v_scale, int32_t hints, void* workspace, size_t workspace_bytes,
    void* stream);

/* Bytes of the static scratch used by paged_attention_forward_static_ws. */
size_t paged_attention_static_workspace_bytes(void);

/* Message for the last non-OK status returned on this thread ("" if none). */
const char* pkv_last_error(void);

/*
 * pkv_device_errors - read (and with clear != 0, reset) the sticky device
 * error word of the current device (PKV_DEVERR_* bits).  Synchronises the
 * device.  Returns PKV_OK and stores the word in *flags.
 */
pkv_status pkv_device_errors(int32_t* flags, int32_t clear);

/*
 * pkv_set_profile_events - instrumentation for benchmarks.  With both
 * arguments non-NULL (cudaEvent_t handles), later paged_attention_forward
 * calls made on this thread record `start` on their stream right before the
 * first attention kernel (after the planner) and `stop` right after the last
 * one (before the split merge), so the attention kernels can be timed alone
 * with cudaEventElapsedTime.  NULL, NULL turns it off.  The events stay the
 * caller's.
 */
void pkv_set_profile_events(void* start, void* stop);

/*
 * pkv_set_profile_mid_event - with profile events set, later forward calls on
 * this thread also record `mid` (a cudaEvent_t) right after the multi-token
 * tensor-core kernel's launch, before the decode-shaped kernel's, so that the
 * former can be timed alone (start .. mid; start .. mid is empty when it does
 * not launch).  The event sits between the two launches, so a call that runs
 * both side by side runs them one after the other while it is set.  NULL
 * turns it off.  The event stays the caller's.
 */
void pkv_set_profile_mid_event(void* mid);

/*
 * pkv_event_elapsed_ms - milliseconds between two recorded events
 * (cudaEventElapsedTime), for events recorded by this library.  Returns
 * PKV_ERR_CUDA if either has not completed.
 */
pkv_status pkv_event_elapsed_ms(void* start, void* stop, float* ms);

/*
 * pkv_debug_fault - testing hook for the bounded in-kernel waits (no
 * counterpart on the source pages).  Arms the next paged_attention_forward /
 * _fp8kv call made on this thread, and only that call:
 *   wait_ns     > 0: every bounded wait of its attention kernels gives up
 *               after wait_ns nanoseconds instead of 2 s;
 *   fault_tile  > 0: in the first CTA of its decode-shaped attention kernel
 *               the K/V producer skips the loads of its fault_tile-th key tile
 *               (counting from 1), so the waits for that tile run out.
 * The kernel then sets PKV_DEVERR_TIMEOUT, every role of the CTA leaves
 * (tensor memory freed, copies in flight awaited) and the call's output is
 * unspecified; the device and later calls are unaffected.  (0, 0) disarms.
 * Returns PKV_ERR_INVALID_ARG for negative arguments.
 */
pkv_status pkv_debug_fault(int32_t fault_tile, int64_t wait_ns);

/* Library version string, e.g. "paged_kv 0.1.0 sm_103a". */
const char* pkv_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PAGED_KV_H_ */
