/*
 * mk_kv.h -- paged-KV block allocator for continuous batching (host memory only).
 *
 * The decode step reads the KV cache through per-row block tables: row b's position t
 * lives in pool page block_tables[b][t / page_size] ("Inside the megakernel serving engine
 * for North Mini Code": paged attention over ragged sequences, continuous batching).  This
 * allocator owns the page bookkeeping of such a pool: a free list of page ids, sequence
 * slots that hold a length and the pages covering it, and the per-step arrays
 * (seq_lens, block_tables) that mk_decode_step takes.  Page ids are shared by every layer
 * (page p of the pool is page p of each layer's cache).  It allocates no device memory and
 * never touches the cache itself; all calls are host-only, O(pages moved), and not
 * thread-safe (one pool per scheduler thread).
 *
 * Free-list order: pages are taken from its head and returned to its tail, in page order,
 * so a given sequence of calls always yields the same page assignment.
 *
 * Return codes are those of mk.h (MK_OK, MK_ERR_INVALID_ARG, MK_ERR_OOM); mk_last_error()
 * describes a failure.  A call that fails changes nothing.
 */
#ifndef MK_KV_H
#define MK_KV_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct mk_kv_pool mk_kv_pool;

/*
 * Create a pool of num_pages pages of page_size tokens, max_slots sequence slots of at most
 * max_pages_per_seq pages each.  order: host int32 [num_pages], a permutation of
 * 0..num_pages-1 giving the initial free-list order, or NULL for ascending.  out receives the
 * pool.  Errors: MK_ERR_INVALID_ARG (non-positive size, NULL out, order not a permutation),
 * MK_ERR_OOM.
 */
int mk_kv_pool_create(int32_t num_pages, int32_t page_size, int32_t max_slots, int32_t max_pages_per_seq,
                      const int32_t* order, mk_kv_pool** out);

/* Free the pool.  NULL is ignored. */
void mk_kv_pool_destroy(mk_kv_pool* pool);

/*
 * Admit a sequence of len >= 1 tokens: take the lowest free slot and ceil(len / page_size)
 * pages from the head of the free list.  slot_out receives the slot.  Errors:
 * MK_ERR_INVALID_ARG (len < 1, more pages than max_pages_per_seq, NULL slot_out), MK_ERR_OOM
 * (no free slot, or fewer free pages than needed).
 */
int mk_kv_admit(mk_kv_pool* pool, int32_t len, int32_t* slot_out);

/*
 * Grow a live slot to len tokens (len >= its length; equal is a no-op), taking pages from
 * the head of the free list for the positions past its last page.  Call it before the step
 * that writes position len-1.  Errors: MK_ERR_INVALID_ARG (slot not live, len smaller than
 * the slot's length or past max_pages_per_seq pages), MK_ERR_OOM (not enough free pages).
 */
int mk_kv_reserve(mk_kv_pool* pool, int32_t slot, int32_t len);

/*
 * Release a live slot: its pages go to the tail of the free list in the slot's page order.
 * Errors: MK_ERR_INVALID_ARG (slot not live).
 */
int mk_kv_evict(mk_kv_pool* pool, int32_t slot);

/*
 * The step arrays for n live slots, row i = slots[i]: seq_lens_out[i] = its length;
 * block_tables_out[i * max_pages_per_seq + p] = its page p, -1 past its pages.  Both are host
 * int32 buffers of n and n * max_pages_per_seq entries.  Errors: MK_ERR_INVALID_ARG (n < 0,
 * NULL buffer, slot not live or listed twice).
 */
int mk_kv_fill(const mk_kv_pool* pool, const int32_t* slots, int32_t n, int32_t* seq_lens_out,
               int32_t* block_tables_out);

/* Pages on the free list (-1 for NULL). */
int32_t mk_kv_free_pages(const mk_kv_pool* pool);

/* Length of a slot, or -1 if it is free or out of range. */
int32_t mk_kv_len(const mk_kv_pool* pool, int32_t slot);

#ifdef __cplusplus
}
#endif

#endif /* MK_KV_H */
