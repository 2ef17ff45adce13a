"""INT4 KV cache (KVQuant-style), restated plainly.  Test infrastructure only.

Source: "KV Cache는 왜 LLM 서빙의 핵심인가", section "KVQuant: 마지막 4배".
K is quantized per channel and V per token (K's outliers sit in a few channels,
V's spread varies token by token); the step size of a group is
s_i = (max - min) / (2^b - 1) with b = 4, and a value maps to round(x / s_i).

Readings of what the page leaves open (each one is also a line of the design notes):

* Zero point.  The printed code round(K / s_i) has no offset, yet s_i spans
  max - min, so the codes would not fit 0..15.  Reading: asymmetric codes
  against the group minimum, code = round((x - min) / s), x^ = code * s + min.
* Precision of each step (fixed so that codes are bit-exact by construction):
  (1) lo, hi = float32 min / max of the group (exact for bf16 inputs); a zero
      minimum is taken as +0 (so the stored fp16 min never depends on the sign of zero);
  (2) s32 = (hi - lo) / 15 in float32, round to nearest;
  (3) s16 = fp16(s32), m16 = fp16(lo), both round to nearest even;
  (4) code = clamp(rint_half_even((x - m16) / s16), 0, 15) with float32
      subtract and divide; a group with s16 == 0 gets code 0 everywhere;
  (5) x^ = code * s16 + m16, the exact value (no rounding).  The page fixes the step
      size and the codes; the reconstruction is read as its plain definition, code times
      scale plus minimum, formed exactly (float64 holds it: a 4-bit code times an fp16
      scale plus an fp16 minimum is a multiple of 2^-24 below 2^21).
* Group extent.  V: the head_dim channels of one (token, kv head).  K: one
  channel of one (block, kv head) over the block's block_size tokens.
* Streaming.  A block's per-channel K range is only known once the block is
  full, so the K rows of a sequence's newest, not-yet-full block stay in a bf16
  tail buffer (one per batch row); when a block's last row is appended the whole
  block is quantized.  V is quantized as each token arrives.
* Nibble order.  The head_dim codes of one row are packed 8 channels to a
  little-endian 32-bit word; nibble n (bits 4n..4n+3) of word w holds channel
  8w + (0, 2, 4, 6, 1, 3, 5, 7)[n], i.e. the low 16 bits carry the even
  channels and the high 16 bits the odd ones.
* Metadata.  K: fp16 [num_blocks][n_kv][2][head_dim] = (scale row, min row).
  V: fp16 [num_blocks][n_kv][block_size][2] = (scale, min) per token.
"""
import numpy as np

NIBBLE_CHANNEL = (0, 2, 4, 6, 1, 3, 5, 7)


def quantize_group(x) -> tuple:
    """Codes (uint8 0..15), fp16 scale and fp16 min of one group, steps (1)-(4) above."""
    x = np.asarray(x, dtype=np.float32)
    lo = np.float32(np.float32(x.min()) + np.float32(0.0))     # -0 + 0 = +0
    hi = np.float32(x.max())
    s32 = np.float32(np.float32(hi - lo) / np.float32(15.0))
    s16 = np.float16(s32)
    m16 = np.float16(lo)
    s = np.float32(s16)
    m = np.float32(m16)
    if s == 0:
        return np.zeros(x.shape, dtype=np.uint8), s16, m16
    q = np.rint((x - m) / s)
    return np.clip(q, 0, 15).astype(np.uint8), s16, m16


def quantize_groups(x) -> tuple:
    """quantize_group applied to every group along the last axis at once (same op sequence).

    x: float32 [..., n] -> codes uint8 [..., n], s16 float16 [...], m16 float16 [...].
    """
    x = np.asarray(x, dtype=np.float32)
    lo = (x.min(axis=-1) + np.float32(0.0)).astype(np.float32)
    hi = x.max(axis=-1)
    s32 = ((hi - lo) / np.float32(15.0)).astype(np.float32)
    s16 = s32.astype(np.float16)
    m16 = lo.astype(np.float16)
    s = s16.astype(np.float32)[..., None]
    m = m16.astype(np.float32)[..., None]
    with np.errstate(divide="ignore", invalid="ignore"):
        q = np.rint((x - m) / s)
    q = np.where(s == 0, 0, np.clip(q, 0, 15))
    return q.astype(np.uint8), s16, m16


def dequantize(codes, s16, m16):
    """x^ = code * s + min (step 5), exact, as float64; s16 / m16 broadcast against codes."""
    return (np.asarray(codes, dtype=np.float64) * np.asarray(s16, dtype=np.float64)
            + np.asarray(m16, dtype=np.float64))


def pack_codes(codes) -> np.ndarray:
    """[..., D] codes 0..15 -> [..., D/2] bytes in the word-interleaved nibble order."""
    c = np.asarray(codes, dtype=np.uint32)
    D = c.shape[-1]
    c = c.reshape(c.shape[:-1] + (D // 8, 8))
    word = np.zeros(c.shape[:-1], dtype=np.uint32)
    for n, ch in enumerate(NIBBLE_CHANNEL):
        word |= (c[..., ch] & 0xF) << np.uint32(4 * n)
    by = np.stack([(word >> np.uint32(8 * i)) & np.uint32(0xFF) for i in range(4)], axis=-1)
    return by.astype(np.uint8).reshape(c.shape[:-2] + (D // 2,))


def unpack_codes(packed) -> np.ndarray:
    """Inverse of pack_codes: [..., D/2] bytes -> [..., D] codes."""
    b = np.asarray(packed, dtype=np.uint32)
    Dh = b.shape[-1]
    b = b.reshape(b.shape[:-1] + (Dh // 4, 4))
    word = b[..., 0] | (b[..., 1] << 8) | (b[..., 2] << 16) | (b[..., 3] << 24)
    out = np.zeros(word.shape + (8,), dtype=np.uint8)
    for n, ch in enumerate(NIBBLE_CHANNEL):
        out[..., ch] = (word >> np.uint32(4 * n)) & np.uint32(0xF)
    return out.reshape(word.shape[:-1] + (Dh * 2,))


class Int4Cache:
    """State of an INT4 paged cache: codes, fp16 metadata and per-row bf16 K tails."""

    def __init__(self, num_blocks, n_kv, block_size, head_dim, batch):
        self.bs = block_size
        self.D = head_dim
        self.k_codes = np.zeros((num_blocks, n_kv, block_size, head_dim // 2), np.uint8)
        self.v_codes = np.zeros((num_blocks, n_kv, block_size, head_dim // 2), np.uint8)
        self.k_meta = np.zeros((num_blocks, n_kv, 2, head_dim), np.float16)
        self.v_meta = np.zeros((num_blocks, n_kv, block_size, 2), np.float16)
        self.k_tail = np.zeros((batch, n_kv, block_size, head_dim), np.float64)

    def append(self, k, v, slot_mapping, tail_seq):
        """Quantize-on-append of n tokens; k, v: [n][n_kv][D] (bf16 values as float64).

        Preconditions (the caller's contract): slots are distinct; within one call
        the tokens of a sequence are consecutive entries in logical order, carry
        the same tail_seq, and a sequence starts at row 0 of its first block.
        """
        bs = self.bs
        slots = [int(x) for x in np.asarray(slot_mapping).tolist()]
        tails = [int(x) for x in np.asarray(tail_seq).tolist()]
        k = np.asarray(k, dtype=np.float64)
        v = np.asarray(v, dtype=np.float64)
        n_kv = k.shape[1]
        completed = set()                      # (seq, block) whose last row arrives in this call
        for i, slot in enumerate(slots):
            if slot < 0:
                continue
            blk, row = divmod(slot, bs)
            codes, s16, m16 = quantize_groups(v[i])               # V: per token, every kv head
            self.v_codes[blk, :, row] = pack_codes(codes)
            self.v_meta[blk, :, row, 0] = s16
            self.v_meta[blk, :, row, 1] = m16
            if row == bs - 1:
                completed.add((tails[i], blk))
        latest = {}                                                 # (seq, slot) -> latest in-call token
        for i, slot in enumerate(slots):                            # K: whole blocks
            if slot < 0:
                continue
            latest[(tails[i], slot)] = i
            if slot % bs != bs - 1:
                continue
            blk, seq = slot // bs, tails[i]
            rows = self.k_tail[seq].copy()                          # rows not in this call
            for r in range(bs):
                j = latest.get((seq, blk * bs + r))
                if j is not None:
                    rows[:, r] = k[j]
            codes, s16, m16 = quantize_groups(rows.transpose(0, 2, 1))   # [n_kv][D] groups of bs rows
            self.k_meta[blk, :, 0] = s16
            self.k_meta[blk, :, 1] = m16
            self.k_codes[blk] = pack_codes(codes.transpose(0, 2, 1))
        for i, slot in enumerate(slots):                            # K tail of unfinished blocks
            if slot < 0:
                continue
            blk, row = divmod(slot, bs)
            if (tails[i], blk) not in completed:
                self.k_tail[tails[i], :, row] = k[i]

    def k_rows(self, s, table_row, ctx, g, start=0):
        """Logical K rows start..ctx-1 of kv group g of batch row s: x^ of full blocks, then the
        bf16 tail.  Only the blocks holding those rows are read."""
        bs, D = self.bs, self.D
        full = int(ctx) // bs
        b0 = int(start) // bs
        parts = []
        for i in range(b0, full):
            blk = int(table_row[i])
            codes = unpack_codes(self.k_codes[blk, g])
            parts.append(dequantize(codes, self.k_meta[blk, g, 0][None, :], self.k_meta[blk, g, 1][None, :]))
        if int(ctx) > full * bs:
            parts.append(self.k_tail[s, g, : int(ctx) - full * bs])
        if not parts or int(start) >= int(ctx):
            return np.zeros((0, D))
        rows = np.concatenate([np.asarray(p, dtype=np.float64) for p in parts], axis=0)
        return rows[int(start) - b0 * bs:]

    def v_rows(self, table_row, ctx, g, start=0):
        """Logical V rows start..ctx-1 of kv group g: x^ with per-token scale and min."""
        bs = self.bs
        nb = -(-int(ctx) // bs)
        b0 = int(start) // bs
        parts = []
        for i in range(b0, nb):
            blk = int(table_row[i])
            codes = unpack_codes(self.v_codes[blk, g])
            parts.append(dequantize(codes, self.v_meta[blk, g, :, 0][:, None], self.v_meta[blk, g, :, 1][:, None]))
        if not parts or int(start) >= int(ctx):
            return np.zeros((0, self.D))
        return np.concatenate(parts, axis=0)[int(start) - b0 * bs: int(ctx) - b0 * bs].astype(np.float64)


def paged_decode_attention_int4(q, cache: Int4Cache, block_tables, context_lens, scale, window=0):
    """Decode attention over the dequantized INT4 cache (float64 on the x^ values); with
    window > 0 over the last `window` tokens only (read as for the bf16 cache)."""
    q = np.asarray(q, dtype=np.float64)
    B, n_h, d = q.shape
    n_kv = cache.k_codes.shape[1]
    G = n_h // n_kv
    out = np.zeros((B, n_h, d))
    for s in range(B):
        L = int(context_lens[s])
        if L <= 0:
            continue
        t0 = max(0, L - int(window)) if window > 0 else 0
        for g in range(n_kv):
            K = cache.k_rows(s, block_tables[s], L, g, t0)
            V = cache.v_rows(block_tables[s], L, g, t0)
            for h in range(g * G, (g + 1) * G):
                logits = scale * (K @ q[s, h])
                w = np.exp(logits - logits.max())
                out[s, h] = (w / w.sum()) @ V
    return out
