"""Pins the oracle's CacheBlend steps (CPU only): KV deviation by closed forms and a
scalar brute force, the recompute ratio by the page's formula, selection against a
library sort, fuse against the (pinned) append, and planted mistakes."""
import math

import numpy as np
import pytest

import oracle
from oracle import cacheblend as cb


def _pools(seed, N=6, n_kv=2, bs=4, d=8):
    rng = np.random.default_rng(seed)
    return rng.standard_normal((N, n_kv, bs, d)), rng.standard_normal((N, n_kv, bs, d))


def test_deviation_closed_forms():
    kp, vp = _pools(0)
    bs = 4
    slots = np.array([0, 5, 13, 23])
    k_same = np.stack([kp[s // bs, :, s % bs] for s in slots])
    v_same = np.stack([vp[s // bs, :, s % bs] for s in slots])
    assert not cb.kv_deviation(kp, vp, slots, k_same, v_same, bs).any()
    # one channel of K off by delta: deviation |delta|
    k1 = k_same.copy(); k1[2, 1, 3] += -0.75
    assert cb.kv_deviation(kp, vp, slots, k1, v_same, bs)[2] == 0.75
    # K off by a along one channel and V by b along another: sqrt(a^2 + b^2)
    k2 = k_same.copy(); v2 = v_same.copy()
    k2[1, 0, 0] += 3.0; v2[1, 1, 5] -= 4.0
    assert abs(cb.kv_deviation(kp, vp, slots, k2, v2, bs)[1] - 5.0) < 1e-12
    # homogeneous of degree 1 in the difference
    rng = np.random.default_rng(1)
    dk, dv = rng.standard_normal(k_same.shape), rng.standard_normal(v_same.shape)
    d1 = cb.kv_deviation(kp, vp, slots, k_same + dk, v_same + dv, bs)
    d3 = cb.kv_deviation(kp, vp, slots, k_same - 3 * dk, v_same - 3 * dv, bs)
    assert np.allclose(d3, 3 * d1, rtol=1e-12, atol=0)


def test_deviation_brute_force():
    kp, vp = _pools(2)
    bs = 4
    rng = np.random.default_rng(3)
    slots = rng.permutation(24)[:9]
    kn, vn = rng.standard_normal((9, 2, 8)), rng.standard_normal((9, 2, 8))
    got = cb.kv_deviation(kp, vp, slots, kn, vn, bs)
    for i, s in enumerate(slots):
        terms = [(float(kp[s // bs, g, s % bs, c]) - float(kn[i, g, c])) ** 2 for g in range(2) for c in range(8)]
        terms += [(float(vp[s // bs, g, s % bs, c]) - float(vn[i, g, c])) ** 2 for g in range(2) for c in range(8)]
        assert abs(got[i] - math.sqrt(math.fsum(terms))) <= 1e-12


def test_recompute_ratio_formula():
    # max(15%, ratio where recompute time = load time)
    assert cb.recompute_ratio(10.0, 100.0) == 0.15
    assert cb.recompute_ratio(40.0, 100.0) == 0.4
    assert cb.recompute_ratio(15.0, 100.0) == 0.15
    assert cb.recompute_ratio(150.0, 100.0) == 1.0
    assert cb.select_count(0.15, 512) == 77           # 76.8 rounds up
    assert cb.select_count(0.15, 20) == 3             # exactly 3
    assert cb.select_count(1.0, 7) == 7 and cb.select_count(0.15, 0) == 0


@pytest.mark.parametrize("seed", range(5))
def test_selection_against_a_library_sort(seed):
    rng = np.random.default_rng(seed)
    n = int(rng.integers(1, 300))
    dev = np.round(rng.random(n) * 20) / 4          # many ties
    for k in (0, 1, n // 7, n // 2, n):
        got = cb.select_top(dev, k)
        order = np.lexsort((np.arange(n), -dev))    # by -dev, then index
        assert got == sorted(order[:k].tolist())
        if 0 < k < n:                               # every selected >= every unselected
            sel = set(got)
            assert min(dev[i] for i in sel) >= max(dev[i] for i in range(n) if i not in sel)


def test_segments_and_progressive_filtering():
    rng = np.random.default_rng(7)
    dev = rng.random(100)
    offs = [0, 30, 30, 100]
    got = cb.select_top_segments(dev, offs, [5, 0, 20])
    assert got == cb.select_top(dev[:30], 5) + [30 + i for i in cb.select_top(dev[30:], 20)]
    # layer 1 picks a generous candidate set, layer 2 narrows it: the result is a subset
    cand = cb.select_top(dev, cb.select_count(0.3, 100))
    dev2 = rng.random(len(cand))
    keep = [cand[i] for i in cb.select_top(dev2, cb.select_count(0.15, 100))]
    assert set(keep) <= set(cand) and len(keep) == 15


def test_fuse_equals_append_of_the_selected_rows():
    kp, vp = _pools(4)
    rng = np.random.default_rng(5)
    kn, vn = rng.standard_normal((10, 2, 8)), rng.standard_normal((10, 2, 8))
    rows = [1, 4, 9]
    slots = np.array([22, 3, 17])
    a = cb.fuse(kp, vp, kn, vn, rows, slots, 4)
    b = oracle.kv_append(kp, vp, kn[rows], vn[rows], slots, 4)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_planted_mistakes_are_caught():
    dev = np.array([0.5, 3.0, 1.0, 3.0, 0.1])
    smallest = sorted(sorted(range(5), key=lambda i: (float(dev[i]), i))[:2])
    assert smallest != cb.select_top(dev, 2) == [1, 3]
    no_floor = lambda load, full: min(1.0, load / full)
    assert no_floor(10.0, 100.0) != cb.recompute_ratio(10.0, 100.0)
