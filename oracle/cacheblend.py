"""CacheBlend's model-free steps, restated plainly.  Test infrastructure only (see the
package header).

Source: "Research Paper Review : CACHE BLEND, Fast Large Language Model Serving for RAG
with Cached Knowledge Fusion":

* section "Methods": a token that needs cross-attention to earlier chunks shows a large
  difference between its precomputed KV and its recomputed KV -- the KV deviation; the
  tokens with the largest deviation are the ones to recompute; a generous candidate set
  chosen on the first layer is narrowed layer by layer to the tokens with the largest
  deviation among the candidates.
* section "System Design": recompute ratio = max(15%, the ratio at which recompute time
  equals load time); the KV cache fusor recomputes the selected tokens and merges the
  updated KV into one KV set.

Readings where the page is silent (each is also a line of the design notes):

* KV deviation of a token: the L2 distance between its precomputed and its recomputed
  K and V, over all kv heads and channels of both (one vector per token), in float64 here.
* Selection: the ceil(ratio * n) candidates with the largest deviation; equal deviations
  are taken lowest token index first; the selected indices are returned in ascending
  order.  The selection is made on the deviation values as given (the GPU's float32
  values when it is checked against the GPU).
* Ratio: recompute time is proportional to the number of recomputed tokens, so the
  ratio at which it equals the load time is load_time / full_recompute_time; the ratio is
  clamped to [0.15, 1].
* Fuse: each selected token's recomputed K and V rows overwrite its rows in the paged
  cache (at its slot); everything else keeps the reused values.
"""
import math

import numpy as np

MIN_RECOMPUTE_RATIO = 0.15


def kv_deviation(k_pool, v_pool, slots, k_new, v_new, block_size):
    """dev[i] = || (K, V) at slots[i] - (k_new[i], v_new[i]) ||_2 over kv heads and channels."""
    out = np.zeros(len(slots))
    for i, slot in enumerate(np.asarray(slots).tolist()):
        blk, row = divmod(int(slot), block_size)
        dk = np.asarray(k_pool[blk, :, row, :], np.float64) - np.asarray(k_new[i], np.float64)
        dv = np.asarray(v_pool[blk, :, row, :], np.float64) - np.asarray(v_new[i], np.float64)
        out[i] = math.sqrt(float(np.sum(dk * dk)) + float(np.sum(dv * dv)))
    return out


def recompute_ratio(load_time, full_recompute_time):
    """max(15%, the ratio whose recompute time equals the load time), at most 1."""
    r = load_time / full_recompute_time if full_recompute_time > 0 else 1.0
    return min(1.0, max(MIN_RECOMPUTE_RATIO, r))


def select_count(ratio, n):
    return min(n, int(math.ceil(ratio * n - 1e-12)))


def select_top(dev, k):
    """Indices of the k largest deviations (ties: lowest index first), ascending."""
    order = sorted(range(len(dev)), key=lambda i: (-float(dev[i]), i))
    return sorted(order[:k])


def select_top_segments(dev, seg_offsets, counts):
    """select_top per segment [seg_offsets[s], seg_offsets[s+1]) with counts[s] tokens;
    returns global indices, ascending."""
    out = []
    for s in range(len(seg_offsets) - 1):
        lo, hi = int(seg_offsets[s]), int(seg_offsets[s + 1])
        out.extend(lo + i for i in select_top(dev[lo:hi], int(counts[s])))
    return out


def fuse(k_pool, v_pool, k_new, v_new, rows, slots, block_size):
    """Copies of the pools with rows[j] of k_new / v_new written at slots[j]."""
    kp = np.array(k_pool, copy=True)
    vp = np.array(v_pool, copy=True)
    for r, slot in zip(np.asarray(rows).tolist(), np.asarray(slots).tolist()):
        blk, row = divmod(int(slot), block_size)
        kp[blk, :, row, :] = k_new[r]
        vp[blk, :, row, :] = v_new[r]
    return kp, vp
