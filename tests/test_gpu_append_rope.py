"""KV append (bit-exact) and RoPE re-rotation on the GPU against the oracle."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_175_gb300 as pkv
import workloads
from gpu_common import DEV, bf16_ulp, err_flag, f64

pytestmark = pytest.mark.gpu


def _bits(t):
    return t.detach().cpu().view(torch.int16).numpy()


@pytest.mark.parametrize("D,BS,n_kv", [(64, 16, 2), (128, 16, 8), (128, 32, 1), (128, 64, 32)])
def test_append_is_bit_exact(D, BS, n_kv):
    rng = np.random.default_rng(D + BS + n_kv)
    num_blocks, n_tok = 40, 300
    g = torch.Generator().manual_seed(1)
    kp = torch.randn(num_blocks, n_kv, BS, D, generator=g).to(torch.bfloat16)
    vp = torch.randn(num_blocks, n_kv, BS, D, generator=g).to(torch.bfloat16)
    k = torch.randn(n_tok, n_kv, D, generator=g).to(torch.bfloat16)
    v = torch.randn(n_tok, n_kv, D, generator=g).to(torch.bfloat16)
    slots = rng.choice(num_blocks * BS, size=n_tok, replace=False).astype(np.int64)
    slots[rng.choice(n_tok, size=20, replace=False)] = -1          # padding tokens
    ek, ev = oracle.kv_append(_bits(kp), _bits(vp), _bits(k), _bits(v), slots, BS)
    kd, vd = kp.to(DEV), vp.to(DEV)
    err = err_flag()
    pkv.kv_append(k.to(DEV), v.to(DEV), torch.as_tensor(slots, device=DEV), kd, vd, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert np.array_equal(_bits(kd), ek) and np.array_equal(_bits(vd), ev)


def test_append_bad_slot_is_flagged_and_skipped():
    kp = torch.zeros(4, 2, 16, 64, dtype=torch.bfloat16, device=DEV)
    vp = torch.zeros_like(kp)
    k = torch.ones(2, 2, 64, dtype=torch.bfloat16, device=DEV)
    err = err_flag()
    pkv.kv_append(k, k, torch.tensor([3, 4 * 16 + 5], device=DEV), kp, vp, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == pkv.DEV_BAD_SLOT
    assert float(kp.abs().sum()) == 2 * 64                  # only the good token landed
    assert torch.equal(kp[0, :, 3], torch.ones(2, 64, dtype=torch.bfloat16, device=DEV))


def _rope_case(D, BS, n_kv, seed):
    rng = np.random.default_rng(seed)
    num_blocks = 60
    g = torch.Generator().manual_seed(seed)
    kp = torch.randn(num_blocks, n_kv, BS, D, generator=g).to(torch.bfloat16)
    ids = rng.choice(num_blocks, size=30, replace=False).astype(np.int32)
    deltas = rng.integers(0, 8193, size=30).astype(np.int32)
    deltas[0], deltas[1], deltas[2] = 0, -377, 8192
    return kp, ids, deltas


def _close_ulps(got, ref, ulps):
    d = np.abs(got - ref)
    tol = ulps * bf16_ulp(ref) + 1e-6 * np.abs(ref).max()
    return bool((d <= tol).all()), float((d / np.maximum(bf16_ulp(ref), 1e-30)).max())


# a CTA takes about 32 KB of rows: several small blocks (capped at 8 for the smallest),
# part of one large block, or ranges that straddle two blocks (9 and 5 kv heads)
@pytest.mark.parametrize("D,BS,n_kv", [(64, 16, 2), (64, 16, 1), (128, 16, 1), (128, 32, 32), (128, 16, 9),
                                       (64, 64, 5)])
def test_rope_shift_matches_oracle(D, BS, n_kv):
    kp, ids, deltas = _rope_case(D, BS, n_kv, seed=D + n_kv)
    ref = oracle.rope_shift_k(f64(kp), ids, deltas)
    kd = kp.to(DEV)
    err = err_flag()
    pkv.rope_shift_k(kd, torch.as_tensor(ids, device=DEV), torch.as_tensor(deltas, device=DEV), err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    got = f64(kd)
    ok, worst = _close_ulps(got, ref, 2)
    assert ok, worst
    untouched = np.setdiff1d(np.arange(kp.shape[0]), ids[1:])   # delta 0 and unlisted blocks
    assert np.array_equal(_bits(kd)[untouched], _bits(kp)[untouched])


def test_rope_composition_on_gpu():
    kp, ids, deltas = _rope_case(128, 16, 2, seed=4)
    a = kp.to(DEV)
    b = kp.to(DEV)
    d1, d2 = deltas // 2, deltas - deltas // 2
    t = lambda x: torch.as_tensor(x, device=DEV)
    pkv.rope_shift_k(a, t(ids), t(d1))
    pkv.rope_shift_k(a, t(ids), t(d2))
    pkv.rope_shift_k(b, t(ids), t(deltas))
    torch.cuda.synchronize()
    # two roundings to bf16: the error is bounded by the ulp of the pair's magnitude, not of
    # the (possibly small) component
    x, y = f64(a), f64(b)
    h = x.shape[-1] // 2
    mag = np.sqrt(y[..., :h] ** 2 + y[..., h:] ** 2)
    mag = np.concatenate([mag, mag], axis=-1)
    assert (np.abs(x - y) <= 3 * bf16_ulp(mag) + 1e-30).all()


def test_rope_bad_block_flagged():
    kp = torch.randn(4, 1, 16, 64).to(torch.bfloat16).to(DEV)
    before = kp.clone()
    err = err_flag()
    pkv.rope_shift_k(kp, torch.tensor([9], dtype=torch.int32, device=DEV),
                     torch.tensor([5], dtype=torch.int32, device=DEV), err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == pkv.DEV_BAD_BLOCK and torch.equal(kp, before)


@pytest.mark.parametrize("name", ["mqa_bs16", "mha_bs32"])
def test_rope_full_size_sampled(name):
    w = workloads.make(name, 0)
    kp, _ = workloads.pools_bf16(w, 0, DEV)
    ids, deltas = w.extra["rope_block_ids"], w.extra["rope_deltas"]
    pick = np.random.default_rng(0).choice(len(ids), size=24, replace=False)
    before = f64(kp[torch.as_tensor(ids[pick], device=DEV)])
    pkv.rope_shift_k(kp, torch.as_tensor(ids, device=DEV), torch.as_tensor(deltas, device=DEV))
    after = f64(kp[torch.as_tensor(ids[pick], device=DEV)])
    ref = oracle.rope_shift_k(before, np.arange(len(pick)), deltas[pick])
    ok, worst = _close_ulps(after, ref, 2)
    assert ok, worst


@pytest.mark.parametrize("D,BS,n_kv", [(128, 16, 1), (128, 16, 9)])
def test_rope_bad_block_inside_a_range_is_skipped(D, BS, n_kv):
    # a bad id among listed blocks that share a CTA's range (small blocks) or whose ranges
    # straddle block edges (9 kv heads): the bad block is flagged and skipped, every other
    # listed block is rotated as the oracle rotates it
    kp, ids, deltas = _rope_case(D, BS, n_kv, seed=77 + n_kv)
    bad = ids.copy()
    bad[5] = kp.shape[0] + 3
    keep = np.array([i for i in range(len(ids)) if i != 5])
    ref = oracle.rope_shift_k(f64(kp), ids[keep], deltas[keep])
    kd = kp.to(DEV)
    err = err_flag()
    pkv.rope_shift_k(kd, torch.as_tensor(bad, device=DEV), torch.as_tensor(deltas, device=DEV), err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == pkv.DEV_BAD_BLOCK
    ok, worst = _close_ulps(f64(kd), ref, 2)
    assert ok, worst
    untouched = np.setdiff1d(np.arange(kp.shape[0]), ids[keep][1:])
    assert np.array_equal(_bits(kd)[untouched], _bits(kp)[untouched])
