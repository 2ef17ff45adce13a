"""Pins the oracle's limited attention window (CPU only).

"KV 캐시 시스템 (KV Cache System)", sections "제한된 어텐션 윈도우 크기 (Limited
Attention Window Size)" and "어텐션 윈도우 크기": a layer with a limited window
attends to the last W tokens of its context; blocks that leave the window are
released; max_attention_window is a per-layer list repeated over the layers.
The pins: brute force with scalar loops, the one-token window as a closed form,
a window over a cache rebuilt from only the window's tokens, stale table entries
before the window, the page's own list example, and a planted off-by-one.
"""
import numpy as np
import pytest

import oracle
import workloads

from test_oracle_attention import _tiny


WINDOWS = [1, 5, 15, 16, 17, 40, 100, 300]


@pytest.mark.parametrize("window", WINDOWS)
def test_window_brute_force_tiny(window):
    w, q, kp, vp = _tiny()
    ref = oracle.paged_decode_attention(q, kp, vp, w.block_tables, w.context_lens, w.scale, w.block_size,
                                        window=window)
    brute = np.array(oracle.attention_loops(q.tolist(), kp.tolist(), vp.tolist(), w.block_tables.tolist(),
                                            w.context_lens.tolist(), w.scale, w.block_size, window=window))
    assert np.max(np.abs(ref - brute)) <= 1e-12


def test_one_token_window_returns_the_newest_value_row():
    w, q, kp, vp = _tiny()
    o = oracle.paged_decode_attention(q, kp, vp, w.block_tables, w.context_lens, w.scale, w.block_size, window=1)
    for s in range(w.batch):
        t = int(w.context_lens[s]) - 1
        blk = w.block_tables[s, t // w.block_size]
        for h in range(w.n_h):
            assert np.array_equal(o[s, h], vp[blk, h // w.group, t % w.block_size])


def test_window_at_least_the_context_is_full_attention():
    w, q, kp, vp = _tiny()
    full = oracle.paged_decode_attention(q, kp, vp, w.block_tables, w.context_lens, w.scale, w.block_size)
    big = int(w.context_lens.max())
    o = oracle.paged_decode_attention(q, kp, vp, w.block_tables, w.context_lens, w.scale, w.block_size, window=big)
    assert np.array_equal(o, full)


@pytest.mark.parametrize("window", [3, 16, 33, 70])
def test_window_equals_full_attention_over_a_cache_of_only_the_window(window):
    # rebuild each sequence's window tokens at rows 0.. of fresh blocks (another alignment
    # inside the blocks) and run full attention on that cache
    w, q, kp, vp = _tiny()
    bs = w.block_size
    ref = oracle.paged_decode_attention(q, kp, vp, w.block_tables, w.context_lens, w.scale, bs, window=window)
    for s in range(w.batch):
        L = int(w.context_lens[s])
        t0 = max(0, L - window)
        n = L - t0
        nb = -(-n // bs)
        k2 = np.zeros((nb,) + kp.shape[1:])
        v2 = np.zeros_like(k2)
        for i, t in enumerate(range(t0, L)):
            blk = w.block_tables[s, t // bs]
            k2[i // bs, :, i % bs] = kp[blk, :, t % bs]
            v2[i // bs, :, i % bs] = vp[blk, :, t % bs]
        o = oracle.paged_decode_attention(q[s:s + 1], k2, v2, np.arange(nb)[None, :], np.array([n]), w.scale, bs)
        assert np.max(np.abs(o[0] - ref[s])) <= 1e-12


def test_blocks_before_the_window_are_never_read():
    w, q, kp, vp = _tiny()
    window = 20
    ref = oracle.paged_decode_attention(q, kp, vp, w.block_tables, w.context_lens, w.scale, w.block_size,
                                        window=window)
    bt = w.block_tables.copy()
    for s in range(w.batch):
        b0 = max(0, int(w.context_lens[s]) - window) // w.block_size
        bt[s, :b0] = 10 ** 6                       # released blocks: no longer valid ids
    o = oracle.paged_decode_attention(q, kp, vp, bt, w.context_lens, w.scale, w.block_size, window=window)
    assert np.array_equal(o, ref)


def test_layer_windows_repeat_the_list():
    # the page's examples: all-full layers with [4096]; alternating full / 256-window with [4096, 256]
    assert oracle.layer_windows([4096], 4) == [4096] * 4
    assert oracle.layer_windows([4096, 256], 6) == [4096, 256, 4096, 256, 4096, 256]
    assert oracle.layer_windows([4096, 256, 128], 4) == [4096, 256, 128, 4096]


def test_window_start():
    assert oracle.window_start(100, 0) == 0
    assert oracle.window_start(100, 100) == 0
    assert oracle.window_start(100, 30) == 70
    assert oracle.window_start(100, 1) == 99


def test_int4_window_reduces_to_bf16_window_on_exact_data():
    # integer data 0..15 per group quantizes exactly, so windowed INT4 attention must equal
    # the windowed bf16 oracle, including windows that start inside the bf16 tail block
    rng = np.random.default_rng(5)
    bs, D, n_kv, n_h, B = 16, 64, 2, 4, 3
    ctx = np.array([3 * bs, 2 * bs + 7, bs + 1])
    table = np.array([[0, 3, 6, -1], [5, 1, 2, -1], [4, 7, -1, -1]])
    nblk = 8
    kpool = np.zeros((nblk, n_kv, bs, D)); vpool = np.zeros_like(kpool)
    cache = oracle.Int4Cache(nblk, n_kv, bs, D, batch=B)
    for s in range(B):
        L = int(ctx[s])
        k = rng.integers(0, 16, size=(L, n_kv, D)).astype(np.float64)
        v = rng.integers(0, 16, size=(L, n_kv, D)).astype(np.float64)
        k[0::bs] = 0; k[1::bs] = 15
        v[:, :, 0] = 0; v[:, :, 1] = 15
        slots = table[s, np.arange(L) // bs] * bs + np.arange(L) % bs
        cache.append(k, v, slots, np.full(L, s))
        for t in range(L):
            kpool[slots[t] // bs, :, slots[t] % bs] = k[t]
            vpool[slots[t] // bs, :, slots[t] % bs] = v[t]
    q = oracle.round_bf16(rng.standard_normal((B, n_h, D)) * 0.1)
    for window in (1, 3, 8, 17, 20, 40, 100):
        a = oracle.paged_decode_attention_int4(q, cache, table, ctx, 0.125, window=window)
        b = oracle.paged_decode_attention(q, kpool, vpool, table, ctx, 0.125, bs, window=window)
        assert np.max(np.abs(a - b)) <= 1e-12, window


def test_planted_off_by_one_window_is_caught():
    # a window that keeps one token too many (start = L - W - 1) must fail the brute-force pin
    w, q, kp, vp = _tiny()
    window = 9
    ctx_plus = w.context_lens
    bad = np.zeros_like(q)
    for s in range(w.batch):
        L = int(ctx_plus[s])
        t0 = max(0, L - window - 1)
        for h in range(w.n_h):
            g = h // w.group
            K = oracle.gather_sequence(kp, w.block_tables[s], L, g, w.block_size, t0)
            V = oracle.gather_sequence(vp, w.block_tables[s], L, g, w.block_size, t0)
            bad[s, h] = oracle.attention_weights(q[s, h], K, w.scale) @ V
    brute = np.array(oracle.attention_loops(q.tolist(), kp.tolist(), vp.tolist(), w.block_tables.tolist(),
                                            w.context_lens.tolist(), w.scale, w.block_size, window=window))
    assert np.max(np.abs(bad - brute)) > 1e-6
