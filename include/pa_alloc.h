/*
 * pa_alloc.h -- host-side block manager for the paged KV cache (libpa.so).
 *
 * A pool of num_blocks physical blocks of block_size token slots, handed out
 * to sequences through block tables that the CALLER holds (plain int32
 * arrays in host memory). The allocator keeps, per block, a reference count
 * (how many tables name it), the token ids written into it and, for full
 * prompt blocks, a chained hash. Everything here runs on the host: no entry
 * point touches device memory or a stream. The device half of copy-on-write
 * is pa_block_copy in pa.h.
 *
 * What it implements ([F] = "LLM 推理底层：KV Cache 显存几何、GQA/MLA 压缩与
 * PagedAttention 调度", section "Prefix Caching 与 Copy-on-Write" and its
 * block-allocator reference; [T] = "KV Cache 显存管理全景", 考点 4 and 5):
 *  - Prefix caching. Full block k of a prompt is named by
 *        H_k = Hash(H_{k-1}, token ids of block k),   H_{-1} = 0,
 *    Hash = BLAKE2b with an 8-byte digest (RFC 7693) over H_{k-1} as 8
 *    little-endian bytes followed by each token id as 4 little-endian bytes;
 *    the digest is read as a little-endian uint64. A new prompt looks up
 *    H_0, H_1, ... in order; a hit shares the cached block (reference count
 *    + 1, block_size tokens reported as cached) and the first miss ends the
 *    lookup for the rest of the prompt.
 *  - Evictable pool. A block whose reference count reaches 0 keeps its data
 *    and hash and joins the tail of an LRU list; new blocks are taken from
 *    the head (least recently released; at creation the list holds every
 *    block in id order). Taking a block drops its hash.
 *  - Appending a decoded token: a full (or missing) last block gets a fresh
 *    block; a partly filled last block shared by several tables is copied
 *    first (copy-on-write) and the caller's table switches to the copy; an
 *    unshared one is written in place.
 *  - Fork: a branch of beam search or parallel sampling shares its parent's
 *    blocks; each block's reference count rises by one ([T] 考点 4).
 *  - Only prompt blocks are hashed, as in [F]'s reference.
 *
 * Error behaviour: every entry point either succeeds or returns an error and
 * leaves the allocator unchanged, except pa_allocator_append_slots, which
 * reports how many sequences it finished (those stay done). Errors:
 * PA_ERR_NULL (a required pointer is NULL), PA_ERR_SHAPE (a negative count
 * or token id, or a table capacity too small for the result),
 * PA_ERR_OUT_OF_BLOCKS, PA_ERR_STATE. The allocator is not thread-safe: one
 * caller thread at a time.
 */
#ifndef PA_ALLOC_H_
#define PA_ALLOC_H_

#include <stdint.h>

#include "pa.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct pa_allocator pa_allocator; /* opaque; owned by the caller */

/* Create an allocator over num_blocks >= 1 blocks of block_size >= 1 slots.
 * *out receives the handle (release with pa_allocator_destroy). */
pa_status pa_allocator_create(int64_t num_blocks, int32_t block_size, pa_allocator **out);
void pa_allocator_destroy(pa_allocator *a);

/*
 * Block table for a new prompt of n_tokens >= 0 token ids (host array).
 *   block_table   host int32 [capacity], receives ceil(n_tokens / block_size)
 *                 block ids
 *   n_blocks      receives that count
 *   cached_tokens receives block_size x the number of prefix-cache hits (the
 *                 tokens whose K/V are already in the pool and need no
 *                 prefill)
 * Token ids must be >= 0. The call first counts its hits without changing
 * anything; if the free blocks (less the hit blocks sitting in the pool)
 * cannot hold the rest, it returns PA_ERR_OUT_OF_BLOCKS and changes nothing.
 */
pa_status pa_allocator_allocate_prompt(pa_allocator *a, const int32_t *token_ids,
                                       int32_t n_tokens, int32_t *block_table, int32_t capacity,
                                       int32_t *n_blocks, int32_t *cached_tokens);

/*
 * Append one decoded token to each of num_seqs sequences, in order.
 *   block_tables  host int32 [num_seqs][capacity], row i holds n_blocks[i]
 *                 valid entries; rows are updated in place (a new block is
 *                 appended, or the last entry switches to its copy)
 *   n_blocks      host int32 [num_seqs], updated
 *   token_ids     host int32 [num_seqs], ids >= 0
 *   slots         host int64 [num_seqs], receives block * block_size + offset
 *                 of each new token (the slot pa_cache_write takes)
 *   cow_pairs     host int32 [num_seqs][2], receives the (source,
 *                 destination) blocks to copy with pa_block_copy, one pair per
 *                 copy-on-write, in sequence order
 *   num_cow       receives the number of pairs written
 *   num_done      receives the number of sequences finished
 * Sequences are processed one after another, so when branches share a tail,
 * all but the last one to append copy it and the last one writes in place.
 * Sequence i is checked before it changes anything; on an error the
 * sequences before it stay done and *num_done = i.
 */
pa_status pa_allocator_append_slots(pa_allocator *a, int32_t *block_tables, int32_t capacity,
                                    int32_t *n_blocks, const int32_t *token_ids,
                                    int32_t num_seqs, int64_t *slots, int32_t *cow_pairs,
                                    int32_t *num_cow, int32_t *num_done);

/* Share every block of a table with a new holder (reference count + 1). */
pa_status pa_allocator_fork(pa_allocator *a, const int32_t *block_table, int32_t n_blocks);

/* Release a table: every block's reference count - 1; blocks that reach 0
 * join the tail of the LRU pool in table order. */
pa_status pa_allocator_free(pa_allocator *a, const int32_t *block_table, int32_t n_blocks);

/* Blocks in the evictable pool (reference count 0). */
int64_t pa_allocator_num_free(const pa_allocator *a);

/* State of one block: reference count, filled slots, and the chained hash
 * (*has_hash = 0 when the block has none). Any output may be NULL. */
pa_status pa_allocator_block_info(const pa_allocator *a, int64_t block, int32_t *ref_count,
                                  int32_t *num_tokens, uint64_t *hash, int32_t *has_hash);

/* The pool's blocks from least to most recently released; writes at most
 * capacity ids and sets *n to the pool size. */
pa_status pa_allocator_free_order(const pa_allocator *a, int32_t *out, int64_t capacity,
                                  int64_t *n);

/* H = BLAKE2b-64(parent as 8 LE bytes || each of n token ids as 4 LE bytes):
 * one link of the chained block hash above (n >= 0, ids >= 0). */
uint64_t pa_block_hash(uint64_t parent, const int32_t *token_ids, int32_t n);

#ifdef __cplusplus
}
#endif

#endif /* PA_ALLOC_H_ */
