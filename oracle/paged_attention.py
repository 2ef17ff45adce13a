"""Paged KV append and paged decode attention, restated plainly in float64.

Test infrastructure only (see the package header).

Sources:

* "KV Cache는 왜 LLM 서빙의 핵심인가", section "KV Cache: O(T²)를 O(T)로": at
  decode step t only the new token's k_t, v_t are computed; they are appended
  to the cached K, V; then attn_t = softmax(q_t K_{1:t}^T / sqrt(d)) V_{1:t}.
  Reading: ``context_lens`` counts the appended token (append, then attend), and
  the caller's ``scale`` stands for 1/sqrt(d) (the configs use 1/sqrt(head_dim)).
* "LLM 서빙과 KV Cache, VLLM", section "PagedAttention": the cache is cut into
  blocks of a fixed number of tokens that need not be contiguous in memory.
  Reading: pool layout [num_blocks][n_kv][block_size][head_dim]; a sequence's
  logical token t lives in physical block block_table[s][t // block_size] at
  row t % block_size.
* "KV Cache는 왜 LLM 서빙의 핵심인가", section "메모리 공식과 GQA의 동기", and
  "KV 캐시 시스템 (KV Cache System)", section "MQA / GQA": n_h query heads share
  n_kv K/V groups (MHA: n_kv = n_h, MQA: n_kv = 1).  Reading: query head h reads
  kv group h // (n_h / n_kv).
* "KV 캐시 시스템 (KV Cache System)", sections "제한된 어텐션 윈도우 크기 (Limited
  Attention Window Size)" and "어텐션 윈도우 크기": a layer may limit its attention
  window, and blocks that fall out of the window are released for reuse.  Reading:
  with a window of W tokens the query attends to the last W tokens of its context,
  [L - W, L), the new token included; W = 0 (or W >= L) is full attention; blocks
  wholly before the window are never read (their table entries may be stale).
"""
import numpy as np


def kv_append(k_pool, v_pool, k, v, slot_mapping, block_size):
    """Return copies of the pools with each new token written at its slot.

    slot = physical block * block_size + row; a negative slot is a padding token
    and is skipped.  Works on any element type (the tests pass raw bf16 bits).
    k, v: [n_tok][n_kv][head_dim].
    """
    kp = np.array(k_pool, copy=True)
    vp = np.array(v_pool, copy=True)
    for i, slot in enumerate(np.asarray(slot_mapping).tolist()):
        if slot < 0:
            continue
        blk, row = divmod(int(slot), block_size)
        kp[blk, :, row, :] = k[i]
        vp[blk, :, row, :] = v[i]
    return kp, vp


def gather_sequence(pool, table_row, ctx, g, block_size, start=0):
    """Logical rows start..ctx-1 of kv group g of one sequence, as a contiguous array.

    Only the blocks holding those rows are read.
    """
    d = pool.shape[-1]
    ctx, start = int(ctx), int(start)
    if start >= ctx:
        return np.zeros((0, d), dtype=np.float64)
    b0, b1 = start // block_size, -(-ctx // block_size)
    tiles = [np.asarray(pool[int(table_row[i]), g], dtype=np.float64) for i in range(b0, b1)]
    return np.concatenate(tiles, axis=0)[start - b0 * block_size: ctx - b0 * block_size]


def window_start(ctx, window):
    """First attended token of a context of ctx tokens under a window of `window` tokens (0 = none)."""
    return max(0, int(ctx) - int(window)) if window > 0 else 0


def layer_windows(max_attention_window, n_layers):
    """Per-layer windows from a max_attention_window list, repeated when shorter than the model."""
    w = list(max_attention_window)
    return [w[i % len(w)] for i in range(n_layers)]


def attention_weights(q_h, K, scale):
    """softmax(scale * K q_h) in float64 (the max is subtracted first; softmax is shift-invariant)."""
    logits = scale * (K @ q_h)
    w = np.exp(logits - logits.max())
    return w / w.sum()


def paged_decode_attention(q, k_pool, v_pool, block_tables, context_lens, scale, block_size, window=0):
    """out[s][h] = softmax(scale * q[s][h] . K_s^T) V_s, K_s / V_s gathered through the block table.

    q: [B][n_h][d]; pools: [num_blocks][n_kv][block_size][d]; returns float64 [B][n_h][d].
    A sequence with context length 0 gives a zero output.  With window > 0, K_s / V_s
    hold only the last `window` tokens.
    """
    q = np.asarray(q, dtype=np.float64)
    B, n_h, d = q.shape
    n_kv = k_pool.shape[1]
    G = n_h // n_kv
    out = np.zeros((B, n_h, d), dtype=np.float64)
    for s in range(B):
        L = int(context_lens[s])
        if L <= 0:
            continue
        t0 = window_start(L, window)
        for g in range(n_kv):
            K = gather_sequence(k_pool, block_tables[s], L, g, block_size, t0)
            V = gather_sequence(v_pool, block_tables[s], L, g, block_size, t0)
            for h in range(g * G, (g + 1) * G):
                out[s, h] = attention_weights(q[s, h], K, scale) @ V
    return out
