"""RoPE re-rotation of reused key chunks.  Test infrastructure only.

Source: "Research Paper Review : CACHE BLEND, Fast Large Language Model Serving
for RAG with Cached Knowledge Fusion", section "Background" (full KV reuse): a
chunk's K/V are precomputed as if the chunk started at position 0; because RoPE
only encodes relative position, the chunk's keys are brought to their real
place by one extra rotation by (real start - 0), applied to every key of the
chunk alike.

Readings (the page names RoPE but not its pairing, base or precision):
rotate pairs (j, j + d/2) for j < d/2 by the angle delta * base^(-2j/d),
base 10000 by default; the oracle works in float64 and rounds the stored key
to bf16 (nearest even) once at the end.
"""
import numpy as np

from .rounding import round_bf16


def rotate(x, delta, base=10000.0):
    """Rotate the last axis of x (float64, length d) by position delta; no rounding."""
    x = np.asarray(x, dtype=np.float64)
    d = x.shape[-1]
    half = d // 2
    theta = float(delta) * np.power(float(base), -2.0 * np.arange(half) / d)
    c, s = np.cos(theta), np.sin(theta)
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * c - x2 * s, x1 * s + x2 * c], axis=-1)


def rope_shift_k(k_pool, block_ids, deltas, base=10000.0):
    """Return a copy of k_pool [num_blocks][n_kv][bs][d] with the listed blocks re-rotated.

    Block block_ids[i] (every kv head, every row) is rotated by deltas[i]; ids are
    distinct.  The result is rounded to bf16 values (float64 array).
    """
    kp = np.array(k_pool, dtype=np.float64, copy=True)
    for b, dl in zip(np.asarray(block_ids).tolist(), np.asarray(deltas).tolist()):
        kp[int(b)] = round_bf16(rotate(kp[int(b)], dl, base))
    return kp
