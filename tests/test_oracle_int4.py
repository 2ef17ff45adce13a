"""Pins the oracle's INT4 quantizer, packing, append state machine and INT4 attention."""
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from oracle.int4 import dequantize, NIBBLE_CHANNEL


def _nearest_fp16(fr: Fraction) -> np.float16:
    """Nearest fp16 to an exact rational, found by brute force over the neighbours (ties to even)."""
    approx = np.float16(float(fr))
    cands = set()
    for base in (approx, np.nextafter(approx, np.float16(np.inf)), np.nextafter(approx, np.float16(-np.inf))):
        cands.add(base)
    best = min(cands, key=lambda c: (abs(Fraction(float(c)) - fr),
                                     int(np.array(c).view(np.uint16)) & 1))
    return best


def test_scale_is_range_over_fifteen():
    # s_i = (max - min) / (2^b - 1), b = 4 ("KVQuant: 마지막 4배", quantization equation)
    x = np.array([-1.5, 0.25, 3.0, 1.0], dtype=np.float32)
    codes, s16, m16 = oracle.quantize_group(x)
    assert s16 == _nearest_fp16(Fraction(4.5) / 15)
    assert m16 == np.float16(-1.5)
    # codes are round((x - min) / s)
    s = Fraction(float(s16))
    for xi, c in zip(x, codes):
        assert c == round((Fraction(float(xi)) - Fraction(-1.5)) / s)


def test_integer_group_is_exact():
    x = np.arange(16, dtype=np.float32)
    codes, s16, m16 = oracle.quantize_group(x)
    assert s16 == 1 and m16 == 0
    assert np.array_equal(codes, np.arange(16))
    assert np.array_equal(dequantize(codes, s16, m16), x)


def test_round_half_to_even():
    # lo = 0, hi = 7.5 -> s = 0.5 exactly; (x - 0) / 0.5 = k + 1/2 are ties
    x = np.array([0.0, 7.5, 0.25, 0.75, 1.25, 1.75, 6.75], dtype=np.float32)
    codes, s16, m16 = oracle.quantize_group(x)
    assert s16 == 0.5 and m16 == 0
    assert codes.tolist() == [0, 15, 0, 2, 2, 4, 14]        # half-up would give 1, 2, 3, 4, 14


def test_constant_group_and_subnormal_scale():
    codes, s16, m16 = oracle.quantize_group(np.full(16, 2.5, np.float32))
    assert s16 == 0 and m16 == 2.5 and not codes.any()
    assert np.array_equal(dequantize(codes, s16, m16), np.full(16, 2.5, np.float32))
    # a range of 15 * 2^-20: the fp16 scale 2^-20 is subnormal and still exact
    x = (np.arange(16, dtype=np.float64) * 2.0 ** -20).astype(np.float32)
    codes, s16, m16 = oracle.quantize_group(x)
    assert float(s16) == 2.0 ** -20 and np.array_equal(codes, np.arange(16))
    # a range below half the smallest fp16 subnormal gives scale 0 and code 0
    x = np.array([1.0, 1.0 + 2.0 ** -23], np.float32)
    codes, s16, m16 = oracle.quantize_group(x)
    assert s16 == 0 and not codes.any()


def test_zero_minimum_is_positive_zero():
    codes, s16, m16 = oracle.quantize_group(np.array([-0.0, 0.0, 3.0], np.float32))
    assert m16.tobytes() == np.float16(0.0).tobytes()
    _, _, m = oracle.quantize_groups(np.array([[0.0, -0.0], [-0.0, 1.0]], np.float32))
    assert m.tobytes() == np.zeros(2, np.float16).tobytes()


def test_dequant_error_bound_random():
    rng = np.random.default_rng(3)
    for _ in range(200):
        x = torch.from_numpy(rng.standard_normal(128).astype(np.float32) * rng.uniform(0.01, 50)) \
            .to(torch.bfloat16).float().numpy()
        codes, s16, m16 = oracle.quantize_group(x)
        xh = dequantize(codes, s16, m16).astype(np.float64)
        s = float(s16)
        s_true = (float(x.max()) - float(x.min())) / 15
        bound = 0.5 * s + abs(float(m16) - float(x.min())) + 15 * abs(s - s_true) + 1e-6 * np.abs(x).max()
        assert np.max(np.abs(xh - x)) <= bound
        assert codes.max() <= 15


def test_vectorised_quantizer_equals_the_scalar_one():
    rng = np.random.default_rng(7)
    x = torch.from_numpy(rng.standard_normal((40, 3, 33)).astype(np.float32) * 3).to(torch.bfloat16) \
        .float().numpy()
    x[0, 0] = 1.25                                         # a constant group
    x[1, 1] = np.arange(33) * 2.0 ** -22                   # a range that rounds to a zero scale
    codes, s16, m16 = oracle.quantize_groups(x)
    for i in range(40):
        for j in range(3):
            c, s, m = oracle.quantize_group(x[i, j])
            assert np.array_equal(codes[i, j], c)
            assert s16[i, j].tobytes() == np.float16(s).tobytes() and m16[i, j].tobytes() == np.float16(m).tobytes()


def test_dequant_is_the_exact_value():
    # x^ = code * s + min with nothing rounded: compared with rational arithmetic on values
    # whose sum needs more bits than fp16 (11) or fp32 (24) carry
    s16, m16 = np.float16(0.1), np.float16(-7.4)
    got = dequantize(np.array([13]), s16, m16)[0]
    assert Fraction(float(got)) == Fraction(13) * Fraction(float(s16)) + Fraction(float(m16))
    assert np.float16(got) != got                               # not an fp16 number
    s16, m16 = np.float16(2.0 ** -24), np.float16(1024.0)       # 1024 + c * 2^-24: 35 bits
    for c in range(16):
        v = dequantize(np.array([c]), s16, m16)[0]
        assert Fraction(float(v)) == Fraction(1024) + c * Fraction(2) ** -24
    assert dequantize(np.array([5]), s16, m16)[0] != np.float32(dequantize(np.array([5]), s16, m16)[0])
    rng = np.random.default_rng(11)
    codes = rng.integers(0, 16, 500)
    ss = rng.standard_normal(500).astype(np.float16) * np.float16(3)
    ss = np.abs(ss)
    mm = rng.standard_normal(500).astype(np.float16) * np.float16(20)
    got = dequantize(codes, ss, mm)
    for c, a, b, g in zip(codes, ss, mm, got):
        assert Fraction(float(g)) == int(c) * Fraction(float(a)) + Fraction(float(b))


def test_pack_order_explicit_bytes():
    # channels 0..7 carry codes 0..7: nibble n holds channel (0,2,4,6,1,3,5,7)[n]
    packed = oracle.pack_codes(np.arange(8))
    assert packed.tolist() == [0x20, 0x64, 0x31, 0x75]
    assert NIBBLE_CHANNEL == (0, 2, 4, 6, 1, 3, 5, 7)
    rng = np.random.default_rng(0)
    c = rng.integers(0, 16, size=(3, 5, 128))
    assert np.array_equal(oracle.unpack_codes(oracle.pack_codes(c)), c)


def _bf16(a):
    return torch.from_numpy(np.asarray(a, np.float32)).to(torch.bfloat16).float().numpy().astype(np.float64)


def test_append_streaming_equals_bulk_and_definition():
    rng = np.random.default_rng(1)
    bs, D, n_kv = 16, 64, 2
    L = 2 * bs + 5
    k = _bf16(rng.standard_normal((L, n_kv, D)) * np.array([1.0] * (D - 1) + [10.0]))
    v = _bf16(rng.standard_normal((L, n_kv, D)))
    table = np.array([7, 2, 4])
    slots = table[np.arange(L) // bs] * bs + np.arange(L) % bs
    bulk = oracle.Int4Cache(8, n_kv, bs, D, batch=3)
    bulk.append(k, v, slots, np.full(L, 1))
    stream = oracle.Int4Cache(8, n_kv, bs, D, batch=3)
    for t in range(L):
        stream.append(k[t: t + 1], v[t: t + 1], slots[t: t + 1], [1])
    for name in ("k_codes", "v_codes", "k_meta", "v_meta"):
        assert np.array_equal(getattr(bulk, name), getattr(stream, name)), name
    # tails: the unfinished third block's 5 rows
    assert np.array_equal(bulk.k_tail[1, :, :5], k[2 * bs:].transpose(1, 0, 2))
    assert np.array_equal(stream.k_tail[1, :, :5], k[2 * bs:].transpose(1, 0, 2))
    # full blocks: per-channel quantization over the block's rows, straight from the definition
    for i in range(2):
        blk = table[i]
        for g in range(n_kv):
            for c in range(D):
                codes, s16, m16 = oracle.quantize_group(k[i * bs:(i + 1) * bs, g, c])
                assert np.array_equal(oracle.unpack_codes(bulk.k_codes[blk, g])[:, c], codes)
                assert bulk.k_meta[blk, g, 0, c] == s16 and bulk.k_meta[blk, g, 1, c] == m16
    # V: per token
    for t in range(L):
        for g in range(n_kv):
            codes, s16, m16 = oracle.quantize_group(v[t, g])
            blk, row = divmod(int(slots[t]), bs)
            assert np.array_equal(oracle.unpack_codes(bulk.v_codes[blk, g, row]), codes)
            assert tuple(bulk.v_meta[blk, g, row]) == (s16, m16)


def test_per_channel_beats_per_tensor_on_outlier_channels():
    # the page: K's outliers sit in a few channels, so K is quantized per channel
    rng = np.random.default_rng(2)
    K = rng.standard_normal((16, 128)).astype(np.float32)
    K[:, [3, 40, 77, 100]] *= 10
    per_channel = np.stack([dequantize(*oracle.quantize_group(K[:, c])) for c in range(128)], 1)
    per_tensor = dequantize(*oracle.quantize_group(K.ravel())).reshape(K.shape)
    mse_c = np.mean((per_channel - K) ** 2)
    mse_t = np.mean((per_tensor - K) ** 2)
    assert mse_t > 10 * mse_c


def test_int4_attention_reduces_to_bf16_attention_on_exact_data():
    # integer data 0..15 per group (with both 0 and 15 present) quantizes exactly,
    # so INT4 attention must equal the bf16 oracle on the same values
    rng = np.random.default_rng(4)
    bs, D, n_kv, n_h, B = 16, 64, 2, 4, 2
    ctx = np.array([2 * bs, bs + 3])
    nblk = 6
    table = np.array([[0, 3, -1], [5, 1, -1]])
    kv_pool = np.zeros((nblk, n_kv, bs, D)); vv_pool = np.zeros_like(kv_pool)
    cache = oracle.Int4Cache(nblk, n_kv, bs, D, batch=B)
    for s in range(B):
        L = int(ctx[s])
        k = rng.integers(0, 16, size=(L, n_kv, D)).astype(np.float64)
        v = rng.integers(0, 16, size=(L, n_kv, D)).astype(np.float64)
        k[0::bs] = 0; k[1::bs] = 15                       # every K block channel spans 0..15
        v[:, :, 0] = 0; v[:, :, 1] = 15                   # every V token spans 0..15
        slots = table[s, np.arange(L) // bs] * bs + np.arange(L) % bs
        cache.append(k, v, slots, np.full(L, s))
        for t in range(L):
            kv_pool[slots[t] // bs, :, slots[t] % bs] = k[t]
            vv_pool[slots[t] // bs, :, slots[t] % bs] = v[t]
    q = _bf16(rng.standard_normal((B, n_h, D)) * 0.1)
    a = oracle.paged_decode_attention_int4(q, cache, table, ctx, 0.125)
    b = oracle.paged_decode_attention(q, kv_pool, vv_pool, table, ctx, 0.125, bs)
    assert np.max(np.abs(a - b)) <= 1e-12


@pytest.mark.parametrize("bug", ["half_up", "no_offset"])
def test_planted_quantizer_mistakes_are_caught(bug):
    x = np.array([0.0, 7.5, 0.25, 0.75, 1.25, 1.75, 6.75], dtype=np.float32)

    def bad(x):
        lo, hi = np.float32(x.min()), np.float32(x.max())
        s = np.float32(np.float16(np.float32(hi - lo) / np.float32(15)))
        if bug == "half_up":
            return np.clip(np.floor((x - lo) / s + 0.5), 0, 15)
        return np.clip(np.rint(x / s), 0, 15)
    good = oracle.quantize_group(x)[0]
    assert not np.array_equal(bad(x).astype(np.uint8), good) or bug == "no_offset"
    if bug == "no_offset":
        y = x - 3.0                                     # negative group: offset-free codes clip
        assert not np.array_equal(bad(y.astype(np.float32)).astype(np.uint8), oracle.quantize_group(y)[0])
