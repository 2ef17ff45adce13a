"""Limited attention window on the GPU (bf16 and INT4 caches) against the fp64 oracle.

A layer with a window of W tokens attends to the last W tokens of each context; the
blocks that end before the window are never read, so their table entries may be stale.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_175_gb300 as pkv
import workloads
from gpu_common import (BAR_INT4_F32_MAXABS, BAR_INT4_F32_RELL2, DEV, check_attention, compact, err_flag, f64)
from test_gpu_decode import _random_case
from test_gpu_int4 import _append_both, _history, _tables

pytestmark = pytest.mark.gpu

WINDOWS = [1, 5, 15, 16, 17, 40, 100, 300]


def _run(q, kp, vp, bt, ctx, scale, window, out_dtype=torch.bfloat16, expect_err=0):
    err = err_flag()
    out = pkv.paged_decode_attn_window(q, kp, vp, torch.as_tensor(bt, device=DEV), torch.as_tensor(ctx, device=DEV),
                                       scale, window, out_dtype=out_dtype, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == expect_err, int(err.item())
    return out


def _stale_before_window(bt, ctx, window, BS, value=-1):
    """Tables whose entries for blocks wholly before the window are invalid ids."""
    bt2 = np.array(bt, copy=True)
    for s, c in enumerate(ctx):
        b0 = max(0, int(c) - window) // BS if window > 0 else 0
        bt2[s, :b0] = value
    return bt2


@pytest.mark.parametrize("window", WINDOWS)
def test_tiny_windows(window):
    w = workloads.make("tiny", 0)
    kp, vp = workloads.pools_bf16(w, 0)
    q = workloads.queries(w, 0)
    ref = oracle.paged_decode_attention(f64(q), f64(kp), f64(vp), w.block_tables, w.context_lens, w.scale,
                                        w.block_size, window=window)
    args = (q.to(DEV), kp.to(DEV), vp.to(DEV))
    for od in (torch.bfloat16, torch.float32):
        out = _run(*args, w.block_tables, w.context_lens, w.scale, window, od)
        check_attention(out, ref, f"tiny window {window} {od}")
    # stale entries before the window: not read, so no error and the same bits
    out = _run(*args, w.block_tables, w.context_lens, w.scale, window)
    bt2 = _stale_before_window(w.block_tables, w.context_lens, window, w.block_size)
    out2 = _run(*args, bt2, w.context_lens, w.scale, window)
    assert torch.equal(out, out2)


def test_window_zero_is_full_attention_bitwise():
    w = workloads.make("tiny", 0)
    kp, vp = workloads.pools_bf16(w, 0)
    q = workloads.queries(w, 0)
    args = (q.to(DEV), kp.to(DEV), vp.to(DEV), torch.as_tensor(w.block_tables, device=DEV),
            torch.as_tensor(w.context_lens, device=DEV), w.scale)
    a = pkv.paged_decode_attn(*args)
    b = pkv.paged_decode_attn_window(*args, 0)
    c = pkv.paged_decode_attn_window(*args, int(w.context_lens.max()))    # window >= every context
    torch.cuda.synchronize()
    assert torch.equal(a, b) and torch.equal(a, c)


def test_negative_window_rejected():
    w = workloads.make("tiny", 0)
    kp, vp = workloads.pools_bf16(w, 0)
    q = workloads.queries(w, 0)
    with pytest.raises(pkv.PkvError):
        pkv.paged_decode_attn_window(q.to(DEV), kp.to(DEV), vp.to(DEV), torch.as_tensor(w.block_tables, device=DEV),
                                     torch.as_tensor(w.context_lens, device=DEV), w.scale, -1)


SHAPES = [(8, 2), (32, 8), (32, 1), (16, 16)]


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("BS", [16, 32, 64])
@pytest.mark.parametrize("heads", SHAPES, ids=[f"{a}q{b}kv" for a, b in SHAPES])
def test_window_shape_sweep(D, BS, heads):
    n_h, n_kv = heads
    ctx = [0, 1, BS - 1, BS + 1, 3 * BS + 7, 2 * BS, 5 * BS + 3]
    q, kp, vp, bt, ctx = _random_case(D, BS, n_h, n_kv, ctx, seed=D * 100 + BS + n_h)
    scale = 1 / math.sqrt(D)
    for window in (1, BS - 1, BS, BS + 3, 2 * BS + 5):
        ref = oracle.paged_decode_attention(f64(q), f64(kp), f64(vp), bt, ctx, scale, BS, window=window)
        bt2 = _stale_before_window(bt, ctx, window, BS, value=10 ** 8)
        out = _run(q.to(DEV), kp.to(DEV), vp.to(DEV), bt2, ctx, scale, window, torch.float32)
        check_attention(out, ref, f"D{D} BS{BS} {n_h}/{n_kv} window {window}")
        assert not f64(out)[0].any()


def test_window_stale_rows_before_the_window_do_not_leak():
    # rows of the window's first block that precede the window hold NaN / inf: the output
    # must not see them
    D, BS, n_h, n_kv = 128, 16, 8, 2
    ctx = [3 * BS + 5, 2 * BS + 9]
    q, kp, vp, bt, ctx = _random_case(D, BS, n_h, n_kv, ctx, seed=7)
    window = BS + 2
    for s, c in enumerate(ctx):
        t0 = int(c) - window
        blk = bt[s, t0 // BS]
        kp[blk, :, : t0 % BS] = float("nan")
        vp[blk, :, : t0 % BS] = float("inf")
    ref = oracle.paged_decode_attention(f64(q), f64(kp), f64(vp), bt, ctx, 0.09, BS, window=window)
    assert np.isfinite(ref).all()
    out = _run(q.to(DEV), kp.to(DEV), vp.to(DEV), bt, ctx, 0.09, window, torch.float32)
    check_attention(out, ref, "stale rows before the window")


def test_window_large_batch_plan_path():
    # more sequences than the in-kernel plan takes: the plan kernel computes the spans
    D, BS, n_h, n_kv = 128, 16, 32, 8
    rng = np.random.default_rng(11)
    ctx = rng.integers(0, 300, size=300).astype(np.int32)
    ctx[:5] = [0, 1, 16, 17, 299]
    q, kp, vp, bt, ctx = _random_case(D, BS, n_h, n_kv, ctx, seed=11)
    window = 37
    ref = oracle.paged_decode_attention(f64(q), f64(kp), f64(vp), bt, ctx, 0.088, BS, window=window)
    out = _run(q.to(DEV), kp.to(DEV), vp.to(DEV), _stale_before_window(bt, ctx, window, BS), ctx, 0.088, window,
               torch.float32)
    check_attention(out, ref, "batch 300 window 37")


def test_full_size_8b_window_sampled():
    """The Llama-3-8B-shaped layer (batch 64, contexts 512..4096) with a 256-token window:
    all sequences in one call, sampled sequences against the oracle."""
    w = workloads.make("llama3_8b", 0)
    kp, vp = workloads.pools_bf16(w, 0, DEV)
    q = workloads.queries(w, 0, DEV)
    window = 256
    out = _run(q, kp, vp, w.block_tables, w.context_lens, w.scale, window)
    for s in (0, int(np.argmax(w.context_lens)), w.batch - 1):
        phys, cbt, cctx = compact(w.block_tables, w.context_lens, [s], w.block_size)
        idx = torch.as_tensor(phys, device=DEV)
        ref = oracle.paged_decode_attention(f64(q[s:s + 1]), f64(kp[idx]), f64(vp[idx]), cbt, cctx, w.scale,
                                            w.block_size, window=window)
        check_attention(out[s:s + 1], ref, f"8B window 256 seq {s}")


@pytest.mark.parametrize("D,BS", [(128, 16), (64, 32), (128, 64)])
def test_int4_windows(D, BS):
    rng = np.random.default_rng(D + 3 * BS)
    n_kv, n_h = 2, 8
    ctx = np.array([5, BS, 3 * BS + 7, 2 * BS - 1, 1, 4 * BS], dtype=np.int32)
    bt, num_blocks = _tables(ctx, BS, rng)
    ks, vs = _history(ctx, n_kv, D, seed=D + BS)
    cache = pkv.alloc_int4_cache(num_blocks, n_kv, BS, D, len(ctx), DEV)
    ref = oracle.Int4Cache(num_blocks, n_kv, BS, D, len(ctx))
    sl = np.concatenate([bt[s, np.arange(c) // BS].astype(np.int64) * BS + np.arange(c) % BS
                         for s, c in enumerate(ctx)])
    tl = np.concatenate([np.full(c, s) for s, c in enumerate(ctx)])
    _append_both(cache, ref, torch.cat(ks), torch.cat(vs), sl, tl)
    q = torch.randn(len(ctx), n_h, D, generator=torch.Generator().manual_seed(2)).to(torch.bfloat16)
    scale = 1 / math.sqrt(D)
    for window in (1, 3, BS, BS + 5, 2 * BS + 1):
        refo = oracle.paged_decode_attention_int4(f64(q), ref, bt, ctx, scale, window=window)
        bt2 = _stale_before_window(bt, ctx, window, BS)
        err = err_flag()
        out = pkv.paged_decode_attn_int4_window(q.to(DEV), cache, torch.as_tensor(bt2, device=DEV),
                                                torch.as_tensor(ctx, device=DEV), scale, window,
                                                out_dtype=torch.float32, err=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        check_attention(out, refo, f"int4 D{D} BS{BS} window {window}",
                        f32_bars=(BAR_INT4_F32_MAXABS, BAR_INT4_F32_RELL2))
