/*
 * pkv.h — C ABI of the GB300 paged KV-cache decode library (libpkv.so).
 *
 * What the library computes, and where the reference pages state it:
 *   - "KV Cache는 왜 LLM 서빙의 핵심인가", section "KV Cache: O(T²)를 O(T)로"
 *     (decode-step listing): each step appends the new token's k_t, v_t to the
 *     cache and computes softmax(q_t K^T / sqrt(d)) V over the whole cache.
 *   - "LLM 서빙과 KV Cache, VLLM", section "PagedAttention": the cache is cut
 *     into fixed-size token blocks that live anywhere in one shared pool.
 *   - "KV Cache는 왜 LLM 서빙의 핵심인가", section "메모리 공식과 GQA의 동기",
 *     and "KV 캐시 시스템 (KV Cache System)", section "MQA / GQA": n_h query
 *     heads share n_kv K/V groups; MHA is n_kv = n_h, MQA is n_kv = 1.
 *   - "KV Cache는 왜 LLM 서빙의 핵심인가", section "KVQuant: 마지막 4배": INT4
 *     K per channel, V per token, step size (max - min) / (2^4 - 1).
 *   - "Research Paper Review : CACHE BLEND ...", section "Background": reused
 *     chunks are brought to their real position by one extra RoPE rotation of
 *     their keys by (real start - 0).
 *
 * Conventions shared by every entry point:
 *   - All tensor pointers are DEVICE pointers owned by the caller.  The library
 *     allocates no device memory and frees nothing; scratch space is passed in
 *     (`workspace`).  Tensors are dense, row-major, in the layouts stated below.
 *   - bf16 / fp16 tensors are passed as `void*` (2-byte elements).
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  Every call
 *     only enqueues work on `stream` and returns; the caller orders calls (e.g.
 *     append before attend) by issuing them on one stream.
 *   - Argument errors are returned synchronously as a negative pkv_status and
 *     nothing is enqueued.  Errors only the GPU can see (a block-table entry or
 *     slot out of range, a context length out of range, a bounded wait that gave
 *     up) set bits in `*err_flag` (a caller-owned device int32, may be NULL): the
 *     offending item is skipped (its block contributes nothing / the token is
 *     not written) and no access goes out of bounds.  The caller clears the flag.
 *   - Pool layout (bf16): [num_blocks][n_kv][block_size][head_dim]; the tile of
 *     one (block, kv head) is contiguous.
 *   - Supported: head_dim in {64, 128}; block_size in {16, 32, 64};
 *     n_h % n_kv == 0 with group n_h / n_kv <= 64.  Other values give PKV_EINVAL.
 *     q, out, pools, codes and workspace must be 16-byte aligned.
 */
#ifndef PKV_H_
#define PKV_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  PKV_OK = 0,
  PKV_EINVAL = -1,   /* bad argument: shape, null pointer, alignment, unsupported size */
  PKV_ERANGE = -2,   /* a size beyond a documented maximum */
  PKV_ECUDA = -3,    /* a CUDA call failed (no device, launch error); see pkv_last_cuda_error() */
  PKV_ENOSPC = -4    /* workspace smaller than pkv_decode_workspace_bytes() */
} pkv_status;

/* Bits ORed into *err_flag by the kernels. */
#define PKV_DEV_BAD_BLOCK 1  /* block_tables entry outside [0, num_blocks): block skipped   */
#define PKV_DEV_BAD_SLOT  2  /* slot >= num_blocks * block_size (or bad tail row): skipped  */
#define PKV_DEV_BAD_CTX   4  /* context_lens[s] < 0 or > max_blocks * block_size: clamped  */
#define PKV_DEV_TIMEOUT   8  /* a bounded wait inside a kernel gave up (about 2 s)          */

/* Output element types of the attention calls. */
#define PKV_OUT_BF16 0
#define PKV_OUT_F32  1

/* Human-readable name of a status. */
const char* pkv_status_str(int status);
/* The last CUDA error code seen by the library on this thread (cudaError_t as int). */
int pkv_last_cuda_error(void);

/*
 * kv_append — write each new token's K and V rows into the pools at its slot.
 * "KV Cache는 왜 LLM 서빙의 핵심인가", section "KV Cache: O(T²)를 O(T)로": the append
 * of the new token's k_t, v_t in each decode step (see file header).
 *   k, v          bf16 [n_tok][n_kv][head_dim]
 *   slot_mapping  int64 [n_tok]; slot = physical block * block_size + row.
 *                 A negative slot is padding and is skipped.  Slots must be distinct.
 *   k_pool,v_pool bf16 [num_blocks][n_kv][block_size][head_dim], updated in place.
 * Bit-exact copy.  A slot >= num_blocks * block_size sets PKV_DEV_BAD_SLOT.
 */
pkv_status pkv_kv_append(const void* k, const void* v, const int64_t* slot_mapping, int n_tok,
                         void* k_pool, void* v_pool, int num_blocks, int block_size, int n_kv,
                         int head_dim, int32_t* err_flag, void* stream);

/*
 * Bytes of workspace pkv_paged_decode_attn (int4 = 0) or pkv_paged_decode_attn_int4
 * (int4 = 1) needs for this shape on the current device.  0 on an invalid shape.
 */
size_t pkv_decode_workspace_bytes(int batch, int n_h, int n_kv, int head_dim, int block_size, int int4);

/*
 * paged_decode_attn — one decode step of attention over a paged bf16 cache.
 * "KV Cache는 왜 LLM 서빙의 핵심인가", section "KV Cache: O(T²)를 O(T)로": the attention
 * of each decode step over the whole cache; PagedAttention blocks; GQA groups (see file
 * header).
 *   q             bf16 [batch][n_h][head_dim]
 *   k_pool,v_pool bf16 [num_blocks][n_kv][block_size][head_dim]
 *   block_tables  int32 [batch][max_blocks]; entry i of row s is the physical block
 *                 holding tokens [i*block_size, (i+1)*block_size) of sequence s.
 *                 Entries past ceil(context_lens[s] / block_size) are not read.
 *   context_lens  int32 [batch]; tokens of sequence s, including the one appended
 *                 this step.  0 gives a zero output row.
 *   scale         multiplies q.k before the softmax (1/sqrt(head_dim) for the usual layer)
 *   out           [batch][n_h][head_dim], bf16 (out_dtype PKV_OUT_BF16, round to
 *                 nearest even) or fp32 (PKV_OUT_F32)
 *   workspace     device scratch of at least pkv_decode_workspace_bytes(..., 0) bytes,
 *                 256-byte aligned; its contents on entry do not matter.
 * Arithmetic: q.k and p.v products in fp32 (tensor-core mma, bf16 inputs, fp32
 * accumulate; p is carried as a bf16 high + low pair), softmax online in fp32.
 * The result depends only on the logical token order, never on which physical
 * blocks hold the tokens.
 * Kernel choice: groups of 17-32 query heads at head_dim 128 run, when the environment
 * variable PKV_ATTN_KERNEL is "tc" at the time of the call, on the fifth-generation tensor
 * cores (tcgen05.mma, 128-token tiles, accumulators in tensor memory, one CTA per SM);
 * otherwise, and for every other shape, on warp-level mma.sync kernels (several CTAs per
 * SM), which measured faster on that shape.  Same arithmetic and bounds either way.
 * The first call of a kernel variant on the device sets its shared-memory attribute and
 * queries occupancy (host-side calls, no stream work); to capture the call into a CUDA
 * graph, make one call of the same shape on the stream before the capture begins.
 */
pkv_status pkv_paged_decode_attn(const void* q, const void* k_pool, const void* v_pool,
                                 const int32_t* block_tables, int max_blocks,
                                 const int32_t* context_lens, float scale, int batch, int n_h,
                                 int n_kv, int head_dim, int block_size, int num_blocks,
                                 void* out, int out_dtype, void* workspace, size_t workspace_bytes,
                                 int32_t* err_flag, void* stream);

/*
 * paged_decode_attn_window — pkv_paged_decode_attn for a layer with a limited
 * attention window.  "KV 캐시 시스템 (KV Cache System)", sections "제한된 어텐션 윈도우
 * 크기 (Limited Attention Window Size)" and "어텐션 윈도우 크기" (max_attention_window).
 *   window        tokens the query attends to: the last `window` tokens of the
 *                 context, [context_lens[s] - window, context_lens[s]); 0 means the
 *                 whole context (the call is then pkv_paged_decode_attn).  Negative:
 *                 PKV_EINVAL.
 *   Table entries of blocks that end before the window are not read (they may hold
 *   released or reused block ids).  Every other argument, the workspace size and the
 *   arithmetic: as pkv_paged_decode_attn.
 */
pkv_status pkv_paged_decode_attn_window(const void* q, const void* k_pool, const void* v_pool,
                                        const int32_t* block_tables, int max_blocks,
                                        const int32_t* context_lens, float scale, int window,
                                        int batch, int n_h, int n_kv, int head_dim, int block_size,
                                        int num_blocks, void* out, int out_dtype, void* workspace,
                                        size_t workspace_bytes, int32_t* err_flag, void* stream);

/*
 * paged_decode_attn_noalloc — pkv_paged_decode_attn without a caller workspace.
 * The reference pages have no counterpart: this entry point exists for callers that
 * cannot allocate device memory when they decode (an engine that gave all free memory
 * to its KV pool, a host program that only receives device pointers from another
 * runtime, code that must not reach an allocator on its hot path).  Its scratch space
 * is a fixed array of PKV_STATIC_SCRATCH_BYTES inside the library, held on every GPU
 * that loads the library until the process exits; the call allocates nothing.
 *   Arguments, layouts, output and device errors: as pkv_paged_decode_attn, minus the
 *   workspace.  Returns PKV_ERANGE, without launching anything, when this shape needs
 *   more scratch than the array holds (pkv_decode_workspace_bytes(..., 0) >
 *   PKV_STATIC_SCRATCH_BYTES).
 *   The first call with a given device current looks up the array's device address
 *   for that device (and looks it up again when the current context has changed, as
 *   after a device reset); make that call before any stream capture.
 *   All calls share the array: calls whose GPU work can overlap (other streams, other
 *   host threads) race on it and must be serialised by the caller.
 */
#define PKV_STATIC_SCRATCH_BYTES (16u * 1024u * 1024u)
pkv_status pkv_paged_decode_attn_noalloc(const void* q, const void* k_pool, const void* v_pool,
                                         const int32_t* block_tables, int max_blocks,
                                         const int32_t* context_lens, float scale, int batch,
                                         int n_h, int n_kv, int head_dim, int block_size,
                                         int num_blocks, void* out, int out_dtype,
                                         int32_t* err_flag, void* stream);

/*
 * layer_window — the attention window of one layer from a max_attention_window list.
 * "KV 캐시 시스템 (KV Cache System)", section "어텐션 윈도우 크기": the list gives one
 * window per layer and is repeated over the layers when it has fewer entries than the
 * model has layers, so layer l takes windows[l % n].  A window at least as long as a
 * context is full attention for it (pkv_paged_decode_attn_window).
 *   windows  host int32 [n], every entry > 0
 * Returns the window (> 0), or -1 for a NULL list, n <= 0, layer < 0 or an entry <= 0.
 */
int pkv_layer_window(const int32_t* windows, int n, int layer);

/*
 * kv_quant_append_int4 — quantize-on-append into an INT4 paged cache.
 * "KVQuant: 마지막 4배": K per channel, V per token, s = (max - min) / 15.
 * Exact op sequence (codes are bit-exact against it):
 *   lo, hi = fp32 min / max of the group (a zero lo is taken as +0);
 *   s32 = (hi - lo) / 15 (fp32, nearest);
 *   s16 = fp16(s32), m16 = fp16(lo) (nearest even);
 *   code = clamp(rint_half_even((x - m16) / s16), 0, 15) (fp32 subtract / divide; the
 *     kernel takes the quotient from the rounded reciprocal away from ties, which gives the
 *     same codes),
 *   code = 0 when s16 == 0; the dequantized value is x^ = code * s16 + m16, exact.
 * Groups: V = the head_dim channels of one (token, kv head); K = one channel of one
 * (block, kv head) over the block's block_size rows.  K rows of a block that is not
 * yet full stay in bf16 in `k_tail`; when a call appends a block's last row, the
 * whole block is quantized from the rows appended earlier in the same call and the
 * tail rows, and the tail is left as it was.
 *   k, v          bf16 [n_tok][n_kv][head_dim]
 *   slot_mapping  int64 [n_tok] (negative = padding); tail_seq int32 [n_tok]: the
 *                 tail row (batch index) of each token's sequence, in [0, tail_rows).
 *   cache         uint8 [num_blocks][n_kv][R], R = pkv_int4_record_bytes(block_size,
 *                 head_dim): one record per (block, kv head), read by the attention
 *                 kernel as one contiguous copy.  Byte offsets inside a record:
 *                   0              K codes  [block_size][head_dim/2]
 *                   bs*d/2         V codes  [block_size][head_dim/2]
 *                   bs*d           K meta   fp16 [2][head_dim]: scale row, then min row
 *                   bs*d + 4d      V meta   fp16 [block_size][2]: (scale, min) per token
 *                 A code row packs 8 channels per little-endian 32-bit word: nibble n of
 *                 word w holds channel 8w + (0,2,4,6,1,3,5,7)[n] (even channels in the
 *                 low half-word).  The K codes and K meta of a block not yet full are
 *                 not defined.
 *   k_tail        bf16 [tail_rows][n_kv][block_size][head_dim].
 * Caller contract: slots distinct; within one call the tokens of a sequence are
 * consecutive entries in logical order with one tail_seq; a sequence starts at
 * row 0 of its first block.  Values must lie within fp16 range.
 * Enqueues two kernels (quantize, then tail update) on `stream`.
 */
pkv_status pkv_kv_quant_append_int4(const void* k, const void* v, const int64_t* slot_mapping,
                                    const int32_t* tail_seq, int n_tok, uint8_t* cache, void* k_tail,
                                    int tail_rows, int num_blocks, int block_size, int n_kv,
                                    int head_dim, int32_t* err_flag, void* stream);

/*
 * Bytes of one (block, kv head) record of the INT4 cache: block_size * head_dim (codes
 * of K and V) + 4 * head_dim (K scale and min rows) + 4 * block_size (V scale and min per
 * token); a multiple of 16.  0 on a shape the INT4 kernels do not take.
 */
size_t pkv_int4_record_bytes(int block_size, int head_dim);

/*
 * paged_decode_attn_int4 — decode attention over the INT4 cache written by
 * pkv_kv_quant_append_int4, equal to the attention over the exact x^ = code * s + m
 * up to fp32 accumulation: no value is dequantized.  Per block, K's per-channel scale is
 * folded into q (q * s as an fp16 pair, high part + exact residual) against the codes as
 * exact small integers, and the block's sum of q * min is one more product; V's per-token
 * scale is folded into the softmax weights (p * s as a bf16 high + low pair) against the
 * codes, and sum_t p_t * (min_t + 8 s_t) is added per head at the end.  The last,
 * unfinished block of sequence s takes its K rows from k_tail[s] (bf16) and its V rows
 * from the codes.
 * Same arguments and output as pkv_paged_decode_attn, with the INT4 cache and the
 * K tail in place of the pools; the batch index is the tail row.  q.k uses fp16 and p.v
 * bf16 tensor-core mma with fp32 accumulation.  q, the tail and every product q_c * s_c
 * must lie in fp16 range.
 */
pkv_status pkv_paged_decode_attn_int4(const void* q, const uint8_t* cache, const void* k_tail,
                                      const int32_t* block_tables,
                                      int max_blocks, const int32_t* context_lens, float scale,
                                      int batch, int n_h, int n_kv, int head_dim, int block_size,
                                      int num_blocks, void* out, int out_dtype, void* workspace,
                                      size_t workspace_bytes, int32_t* err_flag, void* stream);

/*
 * paged_decode_attn_int4_window — pkv_paged_decode_attn_int4 over the last `window`
 * tokens of each context (0: the whole context), with the window read as for
 * pkv_paged_decode_attn_window: the records and table entries of blocks that end before
 * the window are not read.
 */
pkv_status pkv_paged_decode_attn_int4_window(const void* q, const uint8_t* cache, const void* k_tail,
                                             const int32_t* block_tables,
                                             int max_blocks, const int32_t* context_lens, float scale,
                                             int window, int batch, int n_h, int n_kv, int head_dim,
                                             int block_size, int num_blocks, void* out, int out_dtype,
                                             void* workspace, size_t workspace_bytes, int32_t* err_flag,
                                             void* stream);

/*
 * rope_shift_k — re-rotate the keys of reused chunks in place.
 * "Research Paper Review : CACHE BLEND ...", section "Background" (full KV reuse).
 * Every row and kv head of block block_ids[i] is rotated by position deltas[i]:
 * channel pairs (j, j + head_dim/2), angle deltas[i] * rope_base^(-2j/head_dim),
 *   x_j' = x_j cos - x_{j+d/2} sin,  x_{j+d/2}' = x_j sin + x_{j+d/2} cos,
 * angle reduced in fp64, rotation in fp32, stored bf16 (nearest even).
 * A delta of 0 leaves the block untouched.  block_ids must be distinct; an id
 * outside [0, num_blocks) sets PKV_DEV_BAD_BLOCK and is skipped.
 *   k_pool   bf16 [num_blocks][n_kv][block_size][head_dim]
 *   block_ids, deltas  int32 [n_blocks]
 */
pkv_status pkv_rope_shift_k(void* k_pool, const int32_t* block_ids, const int32_t* deltas,
                            int n_blocks, int num_blocks, int n_kv, int block_size, int head_dim,
                            double rope_base, int32_t* err_flag, void* stream);

/*
 * CacheBlend's model-free steps ("Research Paper Review : CACHE BLEND ...", sections
 * "Methods" and "System Design"): the KV deviation of candidate tokens, the selection of
 * the tokens with the largest deviation under the recompute ratio, and the fuse of their
 * recomputed K/V into the cache.  Recomputing K/V needs the model and is the caller's.
 */

/*
 * kv_deviation — dev[i] = L2 distance between the cached K and V of the token at
 * slots[i] and its recomputed rows k_new[i], v_new[i], over all kv heads and channels of
 * K and V together (fp32 accumulation of the squared bf16 differences, then sqrt).
 *   k_pool,v_pool bf16 [num_blocks][n_kv][block_size][head_dim]
 *   slots         int64 [n]
 *   k_new,v_new   bf16 [n][n_kv][head_dim]
 *   dev           fp32 [n] (device)
 * A slot outside the pool sets PKV_DEV_BAD_SLOT and gives dev 0.
 */
pkv_status pkv_kv_deviation(const void* k_pool, const void* v_pool, const int64_t* slots, const void* k_new,
                            const void* v_new, int n, int num_blocks, int block_size, int n_kv, int head_dim,
                            float* dev, int32_t* err_flag, void* stream);

/*
 * select_top — for each segment s = [seg_offsets[s], seg_offsets[s+1]) of dev, the
 * counts[s] elements with the largest values (equal values: lowest index first), written
 * as ascending global indices to out, segment after segment (segment s starts at the sum
 * of the earlier segments' counts).  counts are clamped to [0, segment length].  Values
 * are compared in float32 (NaN above +inf, -0 below +0).
 *   dev fp32 [seg_offsets[n_seg]], seg_offsets int32 [n_seg + 1] (non-decreasing),
 *   counts int32 [n_seg], out int32 [sum of counts]; all device memory.
 */
pkv_status pkv_select_top(const float* dev, const int32_t* seg_offsets, const int32_t* counts, int n_seg,
                          int32_t* out, void* stream);

/*
 * kv_fuse — write the recomputed rows of the selected tokens into the cache:
 * pools[row_slots[rows[j]]] = k_new[rows[j]], v_new[rows[j]] for j < n_sel (rows as
 * pkv_select_top returns them, indexing the candidate rows of k_new / v_new).
 *   k_new,v_new bf16 [n_rows][n_kv][head_dim]; row_slots int64 [n_rows] (the cache slot of
 *   each candidate row); rows int32 [n_sel].
 * A row outside [0, n_rows) or a slot outside the pool sets PKV_DEV_BAD_SLOT and is
 * skipped.  The selected rows' slots must be distinct.
 */
pkv_status pkv_kv_fuse(const void* k_new, const void* v_new, const int64_t* row_slots, int n_rows,
                       const int32_t* rows, int n_sel, void* k_pool, void* v_pool, int num_blocks, int block_size,
                       int n_kv, int head_dim, int32_t* err_flag, void* stream);

/*
 * selftest_wait — exercise the bounded wait that guards every shared-memory ring (the
 * pages have no counterpart: this checks the failure detection of this library).  One
 * thread initialises an mbarrier for one arrival, arrives on it (arrive != 0) or not, and
 * waits for the phase at most limit_us microseconds (1 .. 2 000 000).  A wait that runs out
 * sets PKV_DEV_TIMEOUT in *err_flag (device int32) and the kernel returns normally; the
 * context stays usable.  PKV_EINVAL for a limit out of range or a NULL flag.
 */
pkv_status pkv_selftest_wait(int arrive, int limit_us, int32_t* err_flag, void* stream);

/*
 * probe_read / probe_copy — the HBM bandwidth ceilings the decode kernels are measured
 * against (the pages have no counterpart: these measure the denominator of the roofline
 * fractions).  probe_read streams `bytes` from `buf` with 16-byte loads over a persistent
 * grid (every SM's resident blocks, several loads in flight per thread) and folds the
 * words into a value that is stored to *sink only in a case no data in practice gives;
 * probe_copy copies `bytes` from `src` to `dst` with 16-byte loads and stores.  Time them
 * with events on `stream` over buffers many times the L2: read GB/s = bytes / time,
 * copy GB/s = 2 * bytes / time.
 *   buf, src, dst  device memory, 16-byte aligned; src and dst must not overlap
 *   bytes          a multiple of 16, > 0
 *   sink           device uint32 or NULL
 * PKV_EINVAL on a bad pointer, size or overlap.
 */
pkv_status pkv_probe_read(const void* buf, size_t bytes, uint32_t* sink, void* stream);
pkv_status pkv_probe_copy(const void* src, void* dst, size_t bytes, void* stream);

/* The recompute ratio max(15%, load_time / full_recompute_time), at most 1: the ratio at
 * which recomputing the selected tokens takes as long as loading the layer's KV
 * ("System Design"), recompute time taken as proportional to the tokens recomputed. */
double pkv_recompute_ratio(double load_time, double full_recompute_time);
/* Tokens selected out of n at a ratio: ceil(ratio * n), within [0, n]. */
int pkv_select_count(double ratio, int n);

#ifdef __cplusplus
}
#endif

#endif /* PKV_H_ */
