/*
 * paged_kv_blocks.h - C ABI of the host block manager and the block copy
 * that go with the block-paged KV cache of paged_kv.h.
 *
 * What a block manager does, from the source pages:
 *   - "Paged Attention 基础 - 原理与实现进度", section 3.1 C: a block
 *     allocator that hands out and takes back fixed-size blocks from a free
 *     list, and the per-step [batch_size, max_blocks_per_seq] block table.
 *     Section 1, problem 2: a growing sequence takes one more block and one
 *     more table entry, and nothing already written moves.  Section 1,
 *     problem 3 and section 2: several block tables may name one physical
 *     block (prefix caching: B = [7, 9] shares block 7 of A = [7, 3]).
 *   - "ADR 004: Paged Attention Serving Integration", Decision 5: tables are
 *     keyed by sequence id and cleared by free(seq_id) when a request ends;
 *     Consequences: one update call allocates a fresh sequence or extends an
 *     existing one (prefill and decode alike); Limitations: add_prefix and
 *     try_get_prefix_blocks replay a cached prompt prefix.
 *   - Dao-AILab/flash-attention issue #660: the caller's cache manager copies
 *     and updates the pages; the attention kernels only read them.
 *
 * The manager is host code and owns no device memory: it hands out block
 * ids and slots.  The caller writes K/V through paged_kv_write and copies
 * blocks (copy-on-write) through paged_kv_copy_blocks.  A manager is not
 * thread-safe: serialise the calls on one manager.
 *
 * Policies (the pages leave them open; the library's reference model
 * implements the same ones, so every result below is deterministic):
 *   P1 Free list: initially [num_blocks-1, ..., 1, 0].  Allocation pops its
 *      end (block 0 first); a released block is pushed on the end, so the
 *      block released last is reused first.
 *   P2 A block's reference count is the number of block-table entries that
 *      name it.  A block is free, in use (count > 0), or cached idle (P3).
 *   P3 Prefix cache: full blocks only.  An entry's key is (the parent entry's
 *      id, the block's block_size token ids); the root id is 0 and ids are
 *      never reused, so a key stands for the whole token prefix up to the
 *      block's end.  A cached block whose count drops to 0 stays cached
 *      ("idle", in release order).  Allocation takes the free list first,
 *      then evicts the idle block released longest ago, dropping its entry.
 *   P4 Copy-on-write: when a sequence appends to a partly filled last block
 *      that another table also names, a new block replaces it in this
 *      sequence's table first, and the (src, dst) pair is returned for the
 *      caller to copy before writing the new tokens.
 *   P5 free releases a sequence's blocks from its last to its first, so that
 *      a cached prompt's deepest blocks are evicted first.
 *
 * Errors: PKV_ERR_INVALID_ARG (unknown or duplicate sequence, bad sizes,
 * null pointers, a sequence longer than max_blocks_per_seq blocks) and
 * PKV_ERR_OUT_OF_BLOCKS leave the manager unchanged; pkv_last_error() gives
 * the message.  Sequence ids are any int64 values.
 */
#ifndef PAGED_KV_BLOCKS_H_
#define PAGED_KV_BLOCKS_H_

#include "paged_kv.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct pkv_block_manager pkv_block_manager;

/*
 * pkv_bm_create - a manager of num_blocks blocks of block_size tokens, with
 * at most max_blocks_per_seq blocks per sequence (the width of the block
 * tables it writes).  *out receives the handle; free it with pkv_bm_destroy.
 */
pkv_status pkv_bm_create(int32_t num_blocks, int32_t block_size, int32_t max_blocks_per_seq,
                         pkv_block_manager** out);

/* pkv_bm_destroy - release a manager (NULL is a no-op). */
void pkv_bm_destroy(pkv_block_manager* bm);

/*
 * pkv_bm_update - append num_new_tokens tokens to sequence seq_id, creating
 * it (empty) if unknown ("ADR 004", Consequences: fresh allocation or
 * extension).
 *   slot_mapping  host int64 [num_new_tokens]: the slot of each new token,
 *                 slot = block * block_size + position % block_size (may be
 *                 NULL when num_new_tokens == 0)
 *   copy_pair     host int32 [2]: (src, dst) of the copy-on-write, if any
 *   num_copies    host: 0 or 1
 * The copy must reach the device pool (paged_kv_copy_blocks) before the new
 * tokens are written.
 */
pkv_status pkv_bm_update(pkv_block_manager* bm, int64_t seq_id, int32_t num_new_tokens,
                         int64_t* slot_mapping, int32_t* copy_pair, int32_t* num_copies);

/*
 * pkv_bm_step - one batch step: pkv_bm_update for each sequence in order,
 * all or nothing, and the metadata paged_kv_write and paged_attention_forward
 * take (all host arrays, the caller's):
 *   seq_ids          int64 [num_seqs], distinct
 *   num_new_tokens   int32 [num_seqs], >= 0
 *   slot_mapping     int64 [sum of num_new_tokens], sequences in order
 *   block_tables     int32 [num_seqs, max_blocks_per_seq], -1 past each table's end
 *   context_lens     int32 [num_seqs], tokens after the step
 *   query_start_loc  int32 [num_seqs + 1], prefix sums of num_new_tokens
 *   copies           int32 [num_seqs, 2], the step's (src, dst) copy-on-write pairs
 *   num_copies       number of pairs written to copies
 */
pkv_status pkv_bm_step(pkv_block_manager* bm, const int64_t* seq_ids, const int32_t* num_new_tokens,
                       int32_t num_seqs, int64_t* slot_mapping, int32_t* block_tables,
                       int32_t* context_lens, int32_t* query_start_loc, int32_t* copies,
                       int32_t* num_copies);

/*
 * pkv_bm_free - end sequence seq_id: its table is cleared and each block's
 * count drops by one ("ADR 004", Decision 5).  Blocks left unnamed return to
 * the free list, or stay cached idle if the prefix cache holds them.
 */
pkv_status pkv_bm_free(pkv_block_manager* bm, int64_t seq_id);

/*
 * pkv_bm_fork - a new sequence child_seq_id whose table names the same
 * blocks as parent_seq_id's (parallel sampling, beam search); later appends
 * copy the shared partly filled last block (P4).
 */
pkv_status pkv_bm_fork(pkv_block_manager* bm, int64_t parent_seq_id, int64_t child_seq_id);

/*
 * pkv_bm_add_prefix - make the full blocks of seq_id findable by
 * pkv_bm_try_get_prefix_blocks ("ADR 004", Limitations: add_prefix).
 *   token_ids  host int64 [num_tokens]: all of the sequence's tokens
 *              (num_tokens must equal its length)
 * A block whose token prefix is already cached (on another block) is left
 * uncached; a block cached under a key that no longer chains from the root
 * is re-keyed.
 */
pkv_status pkv_bm_add_prefix(pkv_block_manager* bm, int64_t seq_id, const int64_t* token_ids,
                             int32_t num_tokens);

/*
 * pkv_bm_try_get_prefix_blocks - start sequence seq_id (unknown, or known
 * with no blocks) on the longest chain of cached blocks matching the leading
 * full blocks of its prompt ("ADR 004", Limitations: try_get_prefix_blocks;
 * "Paged Attention 基础", section 1, problem 3: shared prefixes stored once).
 *   token_ids          host int64 [num_tokens], the prompt
 *   num_cached_tokens  out: tokens the attached blocks cover, a multiple of
 *                      block_size and at most num_tokens - 1 (the last
 *                      prompt token is always left to compute, so no step
 *                      writes into a shared block)
 * The sequence's length becomes *num_cached_tokens; pkv_bm_update then adds
 * the rest of the prompt.
 */
pkv_status pkv_bm_try_get_prefix_blocks(pkv_block_manager* bm, int64_t seq_id, const int64_t* token_ids,
                                        int32_t num_tokens, int32_t* num_cached_tokens);

/*
 * pkv_bm_block_table - the table of seq_id: table (host int32
 * [max_blocks_per_seq], -1 past the end), *num_blocks and *num_tokens (any
 * of the three may be NULL).
 */
pkv_status pkv_bm_block_table(const pkv_block_manager* bm, int64_t seq_id, int32_t* table,
                              int32_t* num_blocks, int32_t* num_tokens);

/*
 * pkv_bm_stats - block counts: free (free list), idle (cached, named by no
 * table), used (count > 0), and cached prefix entries.  free + idle + used
 * == num_blocks.  Any pointer may be NULL.
 */
pkv_status pkv_bm_stats(const pkv_block_manager* bm, int32_t* free_blocks, int32_t* idle_blocks,
                        int32_t* used_blocks, int32_t* cached_entries);

/*
 * paged_kv_copy_blocks - the copy-on-write of the device pool: for every
 * pair i and layer l, block copies[i][1] of layer l of k_cache and of v_cache
 * becomes a bit-exact copy of block copies[i][0] (flash-attention issue #660:
 * the cache manager copies pages).
 *   k_cache, v_cache  device, num_layers pools of [num_blocks, block_size,
 *                     num_kv_heads, head_dim], pool l at element offset
 *                     l * layer_stride (0 = num_blocks * block_size *
 *                     num_kv_heads * head_dim, i.e. dense)
 *   copies            HOST int32 [num_copies, 2] (src, dst), as pkv_bm_update and
 *                     pkv_bm_step return them; read before the call returns (the
 *                     pairs travel in the launch parameters, 4000 per launch)
 * Checked on the host before any launch (PKV_ERR_INVALID_ARG): every id in
 * [0, num_blocks), no destination twice, no destination that is also a
 * source (the block manager never produces either).  Pool bases, the block's
 * bytes and the layer stride's bytes must be multiples of 16.  num_copies ==
 * 0 is a no-op.  Asynchronous on `stream`: the copies are ordered before
 * later work on that stream (the step's paged_kv_write).
 */
pkv_status paged_kv_copy_blocks(void* k_cache, void* v_cache, const int32_t* copies, int32_t num_copies,
                                int32_t num_layers, int64_t layer_stride, int64_t num_blocks,
                                int32_t block_size, int32_t num_kv_heads, int32_t head_dim,
                                pkv_dtype dtype, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* PAGED_KV_BLOCKS_H_ */
