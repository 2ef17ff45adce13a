/*
 * pkv_bm.h — host-side KV block manager for the paged cache of pkv.h.
 *
 * Source: "KV 캐시 시스템 (KV Cache System)" (TensorRT-LLM KV cache wiki page):
 *   - "요청 간 재사용 (Reuse Across Requests)": blocks stay reusable across requests until
 *     evicted from the search tree; eviction happens when a free block is needed and is
 *     priority-based LRU, every block carrying a priority 0..100 (100 most important);
 *   - "보존 정책 (Retention Policy)": a request's retention config is a list of token
 *     ranges with priorities; lower-priority blocks are freed first;
 *   - "호스트 메모리로의 오프로딩 (Enable Offloading to Host Memory)": a block may be
 *     offloaded to host memory before it is evicted from GPU memory, stays reusable there,
 *     and is copied back to the GPU when reused; blocks below
 *     secondary_offload_min_priority (default 35) are evicted without offload;
 *   - "제한된 어텐션 윈도우 크기 (Limited Attention Window Size)": blocks that leave the
 *     attention window are released into the search tree.
 * and "LLM 서빙과 KV Cache, VLLM", "PagedAttention": blocks of block_size tokens anywhere
 * in a shared pool, one block table per sequence, slot = block * block_size + row.
 *
 * The manager does host bookkeeping only: it hands out physical block ids (block tables
 * and slots for pkv_kv_append / the attention calls) and records the block copies that
 * offload and onload imply; pkv_copy_blocks (below) performs them on the GPU.
 *
 * Policy (exactly; the readings of what the page leaves open):
 *   - A tree node is one full block of tokens under its parent node (the root for a
 *     sequence's first block), keyed by the parent and the block's token ids.  Only full
 *     blocks enter the tree.  A block is registered when its last row is allocated; if an
 *     identical node exists already the block stays private, and so do the sequence's
 *     later blocks.
 *   - A new request reuses the longest chain of tree nodes matching its full prompt
 *     blocks, at most floor((n_tokens - 1) / block_size) blocks (one token is always left
 *     to compute).  A reused node on the host is copied back (ONLOAD) into a new GPU block.
 *   - Priority of block i: the highest priority among the request's ranges overlapping
 *     tokens [i*bs, (i+1)*bs), else default_priority.  A reused node takes the priority
 *     of the request reusing it.
 *   - Time: a logical clock advanced once per call; a block's time is that of the last
 *     call that allocated, reused or released it.
 *   - A free GPU block is taken lowest id first; with none free, the victim is the
 *     unreferenced cached block with the smallest (priority, time, -depth, block id).  A
 *     victim whose priority is at least offload_min_priority is offloaded (OFFLOAD copy)
 *     if a host slot is free or can be freed by dropping the host block with the smallest
 *     (priority, time, -depth, slot); otherwise it is dropped.  Dropping a node drops its
 *     subtree; blocks of it still held by a sequence leave the tree and stay private.
 *   - Copies must be applied in the order recorded, before the pools are next used.
 *
 * Every function is host-only, not thread-safe for one manager (callers serialise), and
 * allocates host memory only.  Errors: PKV_EINVAL (bad argument, unknown or duplicate
 * sequence id), PKV_ENOSPC (every GPU block is in use by running sequences; the call then
 * changes nothing except evictions it already made, whose copies are still recorded),
 * PKV_ERANGE (an output array is too small).
 */
#ifndef PKV_BM_H_
#define PKV_BM_H_

#include <stdint.h>

#include "pkv.h" /* pkv_status */

#ifdef __cplusplus
extern "C" {
#endif

typedef struct pkv_block_manager pkv_block_manager;

/* Tokens [start, end) of a request get `priority` (0..100); end < 0 means no end. */
typedef struct {
  int32_t start, end, priority;
} pkv_token_range;

/* One recorded copy: kind PKV_COPY_OFFLOAD moves GPU block src to host slot dst,
 * PKV_COPY_ONLOAD moves host slot src to GPU block dst. */
#define PKV_COPY_OFFLOAD 0
#define PKV_COPY_ONLOAD  1
typedef struct {
  int32_t kind, src, dst;
} pkv_block_copy;

/* Counters reported by pkv_bm_counts, in this order. */
#define PKV_BM_N_COUNTS 9 /* free, active, cached, host, reused_tokens, evictions, offloads, onloads, drops */

/* A manager of num_blocks GPU blocks and host_blocks host slots (0: no offload).
 * NULL on an invalid argument (num_blocks < 1, block_size < 1, host_blocks < 0,
 * priorities outside 0..100) or out of memory. */
pkv_block_manager* pkv_bm_create(int num_blocks, int block_size, int host_blocks, int offload_min_priority,
                                 int default_priority);
void pkv_bm_destroy(pkv_block_manager* bm);

/* Start a request with its prompt tokens: reuse what the tree holds, allocate the rest.
 * Writes the ceil(n_tokens / block_size) block ids to table (capacity table_cap) and
 * returns the number of prompt tokens whose K/V are reused (a multiple of block_size;
 * the caller computes and appends tokens from there on), or a negative pkv_status.
 * n_tokens >= 1. */
int pkv_bm_add_sequence(pkv_block_manager* bm, int64_t seq_id, const int32_t* tokens, int n_tokens,
                        const pkv_token_range* ranges, int n_ranges, int32_t* table, int table_cap);

/* Append one generated token to each of n sequences in order (a decode step); slots[i]
 * gets the cache slot of sequence seq_ids[i]'s new token.  Returns PKV_OK, or a negative
 * status with *n_done (if not NULL) the number of sequences served before the failure. */
int pkv_bm_append_tokens(pkv_block_manager* bm, const int64_t* seq_ids, const int32_t* tokens, int n,
                         int64_t* slots, int* n_done);

/* End a request: its registered blocks stay cached in the tree, the others are freed. */
int pkv_bm_release(pkv_block_manager* bm, int64_t seq_id);

/* Release the blocks of a sequence that end before its last `window` tokens (window >= 1)
 * into the tree.  Returns the index of the first block the sequence still holds. */
int pkv_bm_slide_window(pkv_block_manager* bm, int64_t seq_id, int window);

/* Block tables and context lengths of n running sequences for one attention call:
 * tables is [n][max_blocks] (int32, entries past a sequence's blocks and of blocks it
 * released by sliding its window are -1), context_lens [n].  PKV_ERANGE if a sequence has
 * more blocks than max_blocks. */
int pkv_bm_tables(pkv_block_manager* bm, const int64_t* seq_ids, int n, int32_t* tables, int max_blocks,
                  int32_t* context_lens);

/* Move the copies recorded since the last call into out (capacity cap) and return their
 * number; PKV_ERANGE (nothing moved) if more than cap are pending; pkv_bm_pending_copies
 * tells how many. */
int pkv_bm_take_copies(pkv_block_manager* bm, pkv_block_copy* out, int cap);
int pkv_bm_pending_copies(const pkv_block_manager* bm);

/* PKV_BM_N_COUNTS counters (see above). */
void pkv_bm_counts(const pkv_block_manager* bm, int64_t* out);

/*
 * copy_blocks — apply recorded block copies (offload to host, onload back) to a K and a V
 * pool on the GPU ("호스트 메모리로의 오프로딩": offloaded blocks live in host memory and
 * are copied back before reuse).
 *   copies        host array of n pkv_block_copy; the result is that of applying them one
 *                 after another in order
 *   k_pool,v_pool device pools of num_blocks blocks of block_bytes bytes each (for the
 *                 bf16 cache block_bytes = n_kv * block_size * head_dim * 2)
 *   k_host,v_host host pools of host_blocks blocks of block_bytes, in page-locked memory
 *                 the GPU addresses directly (cudaHostAlloc, or registered host memory);
 *                 on a GB300 node the copies cross NVLink-C2C
 * The host splits the list, in order, into waves of copies that touch distinct GPU blocks
 * and host slots; each wave runs as kernel launches of 16-byte vector copies on `stream`.
 * PKV_EINVAL, with nothing launched, for a copy out of range, an unknown kind, pointers
 * not 16-byte aligned, block_bytes not a multiple of 16, or host pools the GPU cannot
 * address.  Ordering against other work is the stream's.
 */
pkv_status pkv_copy_blocks(const pkv_block_copy* copies, int n, void* k_pool, void* v_pool, int num_blocks,
                           void* k_host, void* v_host, int host_blocks, size_t block_bytes, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* PKV_BM_H_ */
