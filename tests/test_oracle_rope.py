"""Pins the oracle's RoPE re-rotation and its bf16 rounding."""
import numpy as np
import pytest
import torch

import oracle


def test_zero_delta_is_identity():
    rng = np.random.default_rng(0)
    x = rng.standard_normal((3, 128))
    assert np.array_equal(oracle.rotate(x, 0), x)


@pytest.mark.parametrize("a,b", [(3, 5), (100, -100), (8000, 192), (1, 8191)])
def test_composition(a, b):
    rng = np.random.default_rng(a * 7 + b)
    x = rng.standard_normal((4, 128))
    two = oracle.rotate(oracle.rotate(x, a), b)
    one = oracle.rotate(x, a + b)
    assert np.max(np.abs(two - one)) <= 1e-12 * max(1, abs(a) + abs(b))


def test_relative_position_invariance():
    # rotating q and k by the same position leaves q.k unchanged: only relative position matters
    rng = np.random.default_rng(1)
    q, k = rng.standard_normal(128), rng.standard_normal(128)
    for p in (1, 37, 4096):
        assert abs(oracle.rotate(q, p) @ oracle.rotate(k, p) - q @ k) <= 1e-10
    # and equals the dot product of the relative shift
    assert abs(oracle.rotate(q, 50) @ oracle.rotate(k, 20) - oracle.rotate(q, 30) @ k) <= 1e-10


def test_complex_multiplication_form():
    # pair (j, j + d/2) as z = x_j + i x_{j+d/2}; rotation multiplies z by exp(i * delta * base^(-2j/d))
    rng = np.random.default_rng(2)
    d = 64
    x = rng.standard_normal(d)
    z = x[: d // 2] + 1j * x[d // 2:]
    theta = 123.0 * 10000.0 ** (-np.arange(d // 2) * 2.0 / d)
    zr = z * np.exp(1j * theta)
    assert np.allclose(oracle.rotate(x, 123), np.concatenate([zr.real, zr.imag]), rtol=0, atol=1e-12)


def test_unit_vector_closed_form():
    d = 128
    e0 = np.zeros(d); e0[0] = 1.0
    r = oracle.rotate(e0, 2.0)                       # channel 0 has frequency base^0 = 1
    assert abs(r[0] - np.cos(2.0)) < 1e-15 and abs(r[64] - np.sin(2.0)) < 1e-15
    assert np.count_nonzero(r) == 2


def test_rope_shift_only_touches_listed_blocks():
    rng = np.random.default_rng(3)
    pool = torch.from_numpy(rng.standard_normal((6, 2, 16, 64)).astype(np.float32)).to(torch.bfloat16) \
        .float().numpy().astype(np.float64)
    out = oracle.rope_shift_k(pool, [4, 1], [7, 300])
    for b in (0, 2, 3, 5):
        assert np.array_equal(out[b], pool[b])
    assert np.array_equal(out[4], oracle.round_bf16(oracle.rotate(pool[4], 7)))
    assert np.array_equal(out[1], oracle.round_bf16(oracle.rotate(pool[1], 300)))


def test_round_bf16_matches_torch_on_float32_values():
    rng = np.random.default_rng(4)
    x = np.concatenate([rng.standard_normal(100000).astype(np.float32) * 10.0 ** rng.integers(-30, 30, 100000),
                        np.array([1e-40, -3e-39, 65504.0, 3.3e38], np.float32)])
    t = torch.from_numpy(x).to(torch.bfloat16).float().numpy().astype(np.float64)
    assert np.array_equal(oracle.round_bf16(x.astype(np.float64)), t)


def test_round_bf16_ties_and_direct_rounding():
    assert oracle.round_bf16(1 + 2.0 ** -8) == 1.0                      # tie, to even
    assert oracle.round_bf16(1 + 3 * 2.0 ** -8) == 1 + 2.0 ** -6        # tie, to even (up)
    assert oracle.round_bf16(1 + 2.0 ** -8 + 2.0 ** -40) == 1 + 2.0 ** -7   # no float32 double rounding
    assert np.isinf(oracle.round_bf16(3.4e38))
