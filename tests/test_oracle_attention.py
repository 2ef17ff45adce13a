"""Pins the oracle's paged decode attention and KV append (CPU only).

Each pin comes from the pages or from mathematics, not from the oracle itself:
brute force with scalar loops, paging as a pure layout change (identity table,
permuted physical blocks), GQA as MHA with replicated K/V, softmax weights
summing to 1, and textbook special cases.  The last tests plant mistakes in a
copy of the oracle and check that the pins catch them.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads

from oracle.paged_attention import gather_sequence, attention_weights


def _f64(t):
    return t.float().numpy().astype(np.float64)


def _tiny(seed=0):
    w = workloads.make("tiny", seed)
    kp, vp = workloads.pools_bf16(w, seed)
    q = workloads.queries(w, seed)
    return w, _f64(q), _f64(kp), _f64(vp)


def test_brute_force_tiny():
    w, q, kp, vp = _tiny()
    ref = oracle.paged_decode_attention(q, kp, vp, w.block_tables, w.context_lens, w.scale, w.block_size)
    bt = w.block_tables.tolist()
    brute = np.array(oracle.attention_loops(q.tolist(), kp.tolist(), vp.tolist(), bt,
                                            w.context_lens.tolist(), w.scale, w.block_size))
    assert np.max(np.abs(ref - brute)) <= 1e-12


def _contiguous_layout(w, kp, vp):
    """Re-lay the same logical cache out with an identity-like table (sequence blocks in order)."""
    nbs = [w.blocks_of(s) for s in range(w.batch)]
    tot = sum(nbs)
    k2 = np.zeros((tot,) + kp.shape[1:])
    v2 = np.zeros_like(k2)
    bt2 = np.full_like(w.block_tables, -1)
    cur = 0
    for s, n in enumerate(nbs):
        for i in range(n):
            k2[cur] = kp[w.block_tables[s, i]]
            v2[cur] = vp[w.block_tables[s, i]]
            bt2[s, i] = cur
            cur += 1
    return k2, v2, bt2


def test_paged_equals_contiguous():
    w, q, kp, vp = _tiny()
    ref = oracle.paged_decode_attention(q, kp, vp, w.block_tables, w.context_lens, w.scale, w.block_size)
    k2, v2, bt2 = _contiguous_layout(w, kp, vp)
    got = oracle.paged_decode_attention(q, k2, v2, bt2, w.context_lens, w.scale, w.block_size)
    assert np.array_equal(ref, got)
    # and against plain dense attention over the concatenated rows, without any table
    for s in range(w.batch):
        L = int(w.context_lens[s])
        start = sum(w.blocks_of(x) for x in range(s)) * w.block_size
        for h in range(w.n_h):
            g = h // w.group
            K = k2[:, g].reshape(-1, w.head_dim)[start: start + L]
            V = v2[:, g].reshape(-1, w.head_dim)[start: start + L]
            logits = w.scale * K @ q[s, h]
            p = np.exp(logits - logits.max())
            assert np.allclose(ref[s, h], (p / p.sum()) @ V, rtol=0, atol=1e-13)


def test_permuted_physical_blocks_give_identical_output():
    w, q, kp, vp = _tiny()
    ref = oracle.paged_decode_attention(q, kp, vp, w.block_tables, w.context_lens, w.scale, w.block_size)
    perm = np.random.default_rng(5).permutation(w.num_blocks)
    inv = np.argsort(perm)
    kp2, vp2 = kp[perm], vp[perm]                 # physical block b moves to position inv[b]
    bt2 = np.where(w.block_tables >= 0, inv[np.maximum(w.block_tables, 0)], -1)
    got = oracle.paged_decode_attention(q, kp2, vp2, bt2, w.context_lens, w.scale, w.block_size)
    assert np.array_equal(ref, got)


def test_gqa_equals_mha_with_replicated_kv():
    w, q, kp, vp = _tiny()
    ref = oracle.paged_decode_attention(q, kp, vp, w.block_tables, w.context_lens, w.scale, w.block_size)
    kr = np.repeat(kp, w.group, axis=1)           # kv head g -> heads g*G .. g*G+G-1
    vr = np.repeat(vp, w.group, axis=1)
    mha = oracle.paged_decode_attention(q, kr, vr, w.block_tables, w.context_lens, w.scale, w.block_size)
    assert np.max(np.abs(ref - mha)) <= 1e-12


def test_weights_sum_to_one_and_are_positive():
    w, q, kp, vp = _tiny()
    for s in range(w.batch):
        K = gather_sequence(kp, w.block_tables[s], w.context_lens[s], 1, w.block_size)
        p = attention_weights(q[s, 5], K, w.scale)
        assert abs(p.sum() - 1.0) <= 1e-12
        assert (p > 0).all()


def test_special_cases():
    w, q, kp, vp = _tiny()
    bt = w.block_tables
    # ctx = 1: the output is the single cached value row
    ctx1 = np.ones(w.batch, dtype=np.int32)
    o = oracle.paged_decode_attention(q, kp, vp, bt, ctx1, w.scale, w.block_size)
    for s in range(w.batch):
        for h in range(w.n_h):
            assert np.array_equal(o[s, h], vp[bt[s, 0], h // w.group, 0])
    # q = 0: uniform weights, the output is the mean of V
    o = oracle.paged_decode_attention(np.zeros_like(q), kp, vp, bt, w.context_lens, w.scale, w.block_size)
    for s in range(w.batch):
        V = gather_sequence(vp, bt[s], w.context_lens[s], 0, w.block_size)
        assert np.allclose(o[s, 0], V.mean(axis=0), rtol=0, atol=1e-13)
    # V == 1: every output is exactly 1
    o = oracle.paged_decode_attention(q, kp, np.ones_like(vp), bt, w.context_lens, w.scale, w.block_size)
    assert np.allclose(o, 1.0, rtol=0, atol=1e-14)
    # ctx = 0: zero output
    o = oracle.paged_decode_attention(q, kp, vp, bt, np.zeros(w.batch, np.int32), w.scale, w.block_size)
    assert not o.any()


def test_two_token_closed_form():
    # two keys: weights are the logistic function of the logit difference
    d = 4
    q = np.zeros((1, 1, d)); q[0, 0, 0] = 1.0
    kp = np.zeros((1, 1, 16, d)); kp[0, 0, 0, 0] = 0.0; kp[0, 0, 1, 0] = 2.0
    vp = np.zeros((1, 1, 16, d)); vp[0, 0, 0, 1] = 1.0; vp[0, 0, 1, 2] = 1.0
    o = oracle.paged_decode_attention(q, kp, vp, np.array([[0]]), np.array([2]), 0.5, 16)
    p1 = 1.0 / (1.0 + math.exp(-1.0))           # logits 0 and 0.5*2 = 1
    assert abs(o[0, 0, 2] - p1) < 1e-15 and abs(o[0, 0, 1] - (1 - p1)) < 1e-15


def test_kv_append_writes_the_token_at_its_logical_position():
    w = workloads.make("tiny", 0)
    kp, vp = workloads.pools_bf16(w, 0)
    kn, vn = workloads.new_tokens(w, 0)
    kb = kp.view(torch.int16).numpy()
    vb = vp.view(torch.int16).numpy()
    slots = workloads.decode_slots(w)
    k2, v2 = oracle.kv_append(kb, vb, kn.view(torch.int16).numpy(), vn.view(torch.int16).numpy(),
                              slots, w.block_size)
    for s in range(w.batch):
        L = int(w.context_lens[s])
        K = gather_sequence(k2, w.block_tables[s], L, 1, w.block_size)
        assert np.array_equal(K[L - 1], kn.view(torch.int16).numpy()[s, 1])
        # every other position is untouched
        K0 = gather_sequence(kb, w.block_tables[s], L, 1, w.block_size)
        assert np.array_equal(K[: L - 1], K0[: L - 1])
    # a negative slot is padding and changes nothing
    k3, v3 = oracle.kv_append(kb, vb, kn.view(torch.int16).numpy(), vn.view(torch.int16).numpy(),
                              -np.ones_like(slots), w.block_size)
    assert np.array_equal(k3, kb) and np.array_equal(v3, vb)
    # exactly batch * n_kv rows changed (when the new rows differ from the old)
    changed = np.any(k2 != kb, axis=-1).sum()
    assert changed == w.batch * w.n_kv


# ---- planted mistakes: a plausible bug in a copy of the oracle must fail a pin ----------

def _attention_variant(bug):
    def f(q, k_pool, v_pool, bt, ctx, scale, bs):
        B, n_h, d = q.shape
        n_kv = k_pool.shape[1]
        G = n_h // n_kv
        out = np.zeros((B, n_h, d))
        for s in range(B):
            L = int(ctx[s])
            for h in range(n_h):
                g = (h % n_kv) if bug == "gqa_map" else h // G
                L2 = L - 1 if bug == "drop_last" else L
                K = gather_sequence(k_pool, bt[s], L2, g, bs)
                V = gather_sequence(v_pool, bt[s], L2, g, bs)
                sc = 1.0 if bug == "no_scale" else scale
                logits = sc * (K @ q[s, h])
                p = np.exp(logits - logits.max())
                out[s, h] = (p / (1.0 if bug == "no_norm" else p.sum())) @ V
        return out
    return f


@pytest.mark.parametrize("bug", ["gqa_map", "drop_last", "no_scale", "no_norm"])
def test_planted_mistake_is_caught_by_brute_force(bug):
    w, q, kp, vp = _tiny()
    got = _attention_variant(bug)(q, kp, vp, w.block_tables, w.context_lens, w.scale, w.block_size)
    brute = np.array(oracle.attention_loops(q.tolist(), kp.tolist(), vp.tolist(), w.block_tables.tolist(),
                                            w.context_lens.tolist(), w.scale, w.block_size))
    assert np.max(np.abs(got - brute)) > 1e-6


def test_planted_transposed_block_index_is_caught_by_permutation_pin():
    # a gather that uses the physical id as the logical index passes an identity table but not a permuted one
    w, q, kp, vp = _tiny()

    def bad_gather(pool, row, ctx, g, bs):
        nb = -(-int(ctx) // bs)
        return np.concatenate([pool[i, g] for i in range(nb)], 0)[: int(ctx)]

    def run(kp_, vp_, bt_):
        out = np.zeros(q.shape)
        for s in range(w.batch):
            for h in range(w.n_h):
                K = bad_gather(kp_, bt_[s], w.context_lens[s], h // w.group, w.block_size)
                V = bad_gather(vp_, bt_[s], w.context_lens[s], h // w.group, w.block_size)
                out[s, h] = attention_weights(q[s, h], K, w.scale) @ V
        return out
    ref = oracle.paged_decode_attention(q, kp, vp, w.block_tables, w.context_lens, w.scale, w.block_size)
    assert np.max(np.abs(run(kp, vp, w.block_tables) - ref)) > 1e-6
