"""The attention kernel on the fifth-generation tensor cores (groups of 17-32 heads at
head_dim 128, selected with PKV_ATTN_KERNEL=tc) against the fp64 oracle: tiles cut by segment and piece ends, windows, stale
NaN / inf rows, bad block ids, the plan-kernel path and bitwise invariance."""
import math

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_175_gb300 as pkv
from gpu_common import DEV, check_attention, err_flag, f64, run_attention

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def tensor_memory_kernel(monkeypatch):
    # the library reads PKV_ATTN_KERNEL at every call: these tests run the tcgen05 kernel
    monkeypatch.setenv("PKV_ATTN_KERNEL", "tc")


def _case(BS, n_h, n_kv, ctx, seed, pool_extra=7):
    rng = np.random.default_rng(seed)
    ctx = np.asarray(ctx, dtype=np.int32)
    nbs = [-(-int(c) // BS) for c in ctx]
    num_blocks = sum(nbs) + pool_extra
    perm = rng.permutation(num_blocks).astype(np.int32)
    bt = np.full((len(ctx), max(1, max(nbs))), -1, dtype=np.int32)
    cur = 0
    for s, n in enumerate(nbs):
        bt[s, :n] = perm[cur:cur + n]
        cur += n
    g = torch.Generator().manual_seed(seed)
    kp = torch.randn(num_blocks, n_kv, BS, 128, generator=g).to(torch.bfloat16)
    vp = torch.randn(num_blocks, n_kv, BS, 128, generator=g).to(torch.bfloat16)
    q = torch.randn(len(ctx), n_h, 128, generator=g).to(torch.bfloat16)
    return q, kp, vp, bt, ctx


HEADS = [(32, 1), (64, 2), (24, 1), (17, 1), (96, 3)]


@pytest.mark.parametrize("BS", [16, 32, 64])
@pytest.mark.parametrize("heads", HEADS, ids=[f"{a}q{b}kv" for a, b in HEADS])
def test_group_sizes_and_ragged_tiles(BS, heads):
    n_h, n_kv = heads
    # contexts ending inside a block, on a block edge, on a 128-token tile edge, one token,
    # empty, and long ones cut into several tiles and pieces
    ctx = [0, 1, BS - 1, 128, 129, 3 * BS + 7, 1000, 4096 + 5]
    q, kp, vp, bt, ctx = _case(BS, n_h, n_kv, ctx, seed=BS * 100 + n_h)
    scale = 1 / math.sqrt(128)
    ref = oracle.paged_decode_attention(f64(q), f64(kp), f64(vp), bt, ctx, scale, BS)
    for od in (torch.bfloat16, torch.float32):
        out = run_attention(q.to(DEV), kp.to(DEV), vp.to(DEV), bt, ctx, scale, od)
        check_attention(out, ref, f"tc BS{BS} {n_h}/{n_kv} {od}")
        assert not f64(out)[0].any()


@pytest.mark.parametrize("BS", [16, 32])
def test_windows(BS):
    q, kp, vp, bt, ctx = _case(BS, 32, 1, [5, 300, 1000, 2048, 77], seed=5 + BS)
    for window in (1, 15, 16, 17, 100, 129, 600):
        ref = oracle.paged_decode_attention(f64(q), f64(kp), f64(vp), bt, ctx, 0.09, BS, window=window)
        err = err_flag()
        out = pkv.paged_decode_attn_window(q.to(DEV), kp.to(DEV), vp.to(DEV), torch.as_tensor(bt, device=DEV),
                                           torch.as_tensor(ctx, device=DEV), 0.09, window, out_dtype=torch.float32,
                                           err=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        check_attention(out, ref, f"tc window {window} BS{BS}")


def test_stale_nan_rows_past_the_context_do_not_leak():
    BS = 16
    q, kp, vp, bt, ctx = _case(BS, 32, 1, [37, 130, 250, 1], seed=21)
    for s, c in enumerate(ctx):
        last = bt[s, (int(c) - 1) // BS]
        r = int(c) % BS
        if r:
            kp[last, :, r:] = float("nan")
            vp[last, :, r:] = float("inf")
    ref = oracle.paged_decode_attention(f64(q), np.nan_to_num(f64(kp)), np.nan_to_num(f64(vp)), bt, ctx, 0.1, BS)
    out = run_attention(q.to(DEV), kp.to(DEV), vp.to(DEV), bt, ctx, 0.1, torch.float32)
    check_attention(out, ref, "tc stale NaN")


def test_bad_block_id_is_flagged_and_skipped():
    BS = 16
    q, kp, vp, bt, ctx = _case(BS, 32, 1, [200, 64], seed=8)
    bad = bt.copy()
    bad[0, 3] = kp.shape[0] + 50
    # the oracle without that block: its 16 tokens removed from sequence 0
    keep = np.ones(200, bool)
    keep[48:64] = False
    k0 = np.concatenate([f64(kp)[bt[0, i // BS], 0, i % BS][None] for i in range(200) if keep[i]])
    v0 = np.concatenate([f64(vp)[bt[0, i // BS], 0, i % BS][None] for i in range(200) if keep[i]])
    out = run_attention(q.to(DEV), kp.to(DEV), vp.to(DEV), bad, ctx, 0.1, torch.float32, expect_err=pkv.DEV_BAD_BLOCK)
    for h in range(32):
        logits = 0.1 * (k0 @ f64(q)[0, h])
        w = np.exp(logits - logits.max())
        ref = (w / w.sum()) @ v0
        got = f64(out)[0, h]
        assert np.abs(got - ref).max() <= 5e-4, h


def test_plan_kernel_path_and_bitwise_permutation():
    BS = 16
    ctx = [3] * 280 + [900, 2049, 17]
    q, kp, vp, bt, ctx = _case(BS, 32, 1, ctx, seed=13, pool_extra=60)
    ref = oracle.paged_decode_attention(f64(q), f64(kp), f64(vp), bt, ctx, 0.1, BS)
    a = run_attention(q.to(DEV), kp.to(DEV), vp.to(DEV), bt, ctx, 0.1, torch.float32)
    check_attention(a, ref, "tc plan kernel")
    perm = np.random.default_rng(2).permutation(kp.shape[0])
    inv = np.argsort(perm)
    bt2 = np.where(bt >= 0, inv[np.maximum(bt, 0)], -1).astype(np.int32)
    b = run_attention(q.to(DEV), kp[perm].to(DEV), vp[perm].to(DEV), bt2, ctx, 0.1, torch.float32)
    assert torch.equal(a, b)
    c = run_attention(q.to(DEV), kp.to(DEV), vp.to(DEV), bt, ctx, 0.1, torch.float32)
    assert torch.equal(a, c)


def test_value_rows_of_ones_give_exactly_one():
    q, kp, vp, bt, ctx = _case(32, 32, 1, [1, 31, 500, 1500], seed=4)
    vp = torch.ones_like(vp)
    out = run_attention(q.to(DEV), kp.to(DEV), vp.to(DEV), bt, ctx, 0.3)
    assert torch.equal(out, torch.ones_like(out))
