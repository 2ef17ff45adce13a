"""Host restatement of the arithmetic the INT4 attention kernel relies on to fold the
scales instead of dequantizing (no GPU): the code encodings are exact, the fp16 high part
plus residual of q * s is exactly q * s, and the two folds are identities of the
reconstruction x^ = code * s + min ("KV Cache는 왜 LLM 서빙의 핵심인가", "KVQuant: 마지막 4배")."""
import numpy as np
import torch

import oracle
from oracle.int4 import dequantize


def _bf16_bits_to_float(bits):
    return torch.tensor(np.asarray(bits, dtype=np.int32).astype(np.int16)).view(torch.bfloat16).float().numpy()


def test_code_encodings_are_exact():
    c = np.arange(16, dtype=np.uint16)
    # K: fp16 0x4c00 | code << 6 is 16 + code (mantissa bits 6..9 under the exponent of 16)
    k = (np.uint16(0x4C00) | (c << 6)).view(np.float16).astype(np.float64)
    assert np.array_equal(k, 16 + c)
    # V: bf16 0x4300 | code is 128 + code; minus 136 (bf16 0x4308) is code - 8, exactly
    v = _bf16_bits_to_float(np.uint16(0x4300) | c)
    assert np.array_equal(v, 128 + c)
    assert _bf16_bits_to_float([0x4308])[0] == 136.0
    assert np.array_equal(v - 136.0, c.astype(np.float64) - 8)


def test_nibble_pair_shifts_land_in_the_mantissa_field():
    # nibble j of a packed word sits at bits 4j (and j + 4 at 16 + 4j); the kernel moves the
    # pair to bits 6..9 / 22..25 by shifting left 6, 2 or right 2, 6
    rng = np.random.default_rng(0)
    for _ in range(200):
        word = int(rng.integers(0, 2 ** 32))
        for j, sh in enumerate((6, 2, -2, -6)):
            x = (word << sh if sh > 0 else word >> -sh) & 0xFFFFFFFF
            x = (x & 0x03C003C0) | 0x4C004C00
            lo = np.array([x & 0xFFFF], np.uint16).view(np.float16)[0]
            hi = np.array([x >> 16], np.uint16).view(np.float16)[0]
            assert lo == 16 + ((word >> (4 * j)) & 15) and hi == 16 + ((word >> (16 + 4 * j)) & 15)


def test_high_part_plus_residual_is_the_exact_product():
    # q is a bf16 value (8 significant bits), s an fp16 scale (11): q * s has at most 19
    # significant bits, so fp16(q s) + fp16(q s - fp16(q s)) is q s exactly while the
    # residual is a normal fp16 number
    rng = np.random.default_rng(1)
    q = torch.from_numpy(rng.standard_normal(20000).astype(np.float32) * 3).to(torch.bfloat16).float().numpy()
    s = (np.abs(rng.standard_normal(20000)) * rng.choice([0.01, 0.3, 4.0], 20000)).astype(np.float16)
    exact = q.astype(np.float64) * s.astype(np.float64)
    hi = exact.astype(np.float16)                       # one rounding of the exact product
    lo = (exact - hi.astype(np.float64)).astype(np.float16)
    normal = np.abs(lo.astype(np.float64)) >= 2.0 ** -14
    assert np.array_equal((hi.astype(np.float64) + lo.astype(np.float64))[normal], exact[normal])
    # where the residual underflows the error is below the smallest fp16 step
    assert np.abs(hi.astype(np.float64) + lo.astype(np.float64) - exact).max() <= 2.0 ** -25


def test_folds_are_identities_of_the_reconstruction():
    rng = np.random.default_rng(2)
    D, n = 128, 48
    x = torch.from_numpy(rng.standard_normal((n, D)).astype(np.float32)).to(torch.bfloat16).float().numpy()
    x[:, 3] *= 10
    q = rng.standard_normal(D)
    p = rng.random(n)
    # K: per-channel groups over the n rows
    ck, sk, mk = oracle.quantize_groups(x.T)
    kh = dequantize(ck.T, sk[None, :], mk[None, :])
    s64, m64 = sk.astype(np.float64), mk.astype(np.float64)
    scores = ((16 + ck.T.astype(np.float64)) @ (q * s64)) + q @ (m64 - 16 * s64)
    assert np.allclose(scores, kh @ q, rtol=0, atol=1e-9)
    # V: per-token groups
    cv, sv, mv = oracle.quantize_groups(x)
    vh = dequantize(cv, sv[:, None], mv[:, None])
    s64, m64 = sv.astype(np.float64), mv.astype(np.float64)
    o = (cv.astype(np.float64) - 8).T @ (p * s64) + p @ (m64 + 8 * s64)
    assert np.allclose(o, vh.T @ p, rtol=0, atol=1e-9)
