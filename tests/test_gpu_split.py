"""Sequences split across CTAs (segments cut by piece boundaries, merged by the split-reduce):
one workspace serves calls of different shapes in any order whatever it holds on entry, and
a segment spread over hundreds of pieces merges to the oracle's result, bit for bit the same
on every call."""
import math

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_175_gb300 as pkv
from gpu_common import DEV, check_attention, err_flag, f64

pytestmark = pytest.mark.gpu


def _case(B, n_h, n_kv, ctx, BS, seed, D=128):
    rng = np.random.default_rng(seed)
    ctx = np.asarray(ctx, dtype=np.int32)
    nbs = [-(-int(c) // BS) for c in ctx]
    num_blocks = sum(nbs) + 5
    perm = rng.permutation(num_blocks).astype(np.int32)
    bt = np.full((B, max(1, max(nbs))), -1, dtype=np.int32)
    cur = 0
    for s, n in enumerate(nbs):
        bt[s, :n] = perm[cur:cur + n]
        cur += n
    g = torch.Generator().manual_seed(seed)
    kp = torch.randn(num_blocks, n_kv, BS, D, generator=g).to(torch.bfloat16)
    vp = torch.randn(num_blocks, n_kv, BS, D, generator=g).to(torch.bfloat16)
    q = torch.randn(B, n_h, D, generator=g).to(torch.bfloat16)
    return q, kp, vp, bt, ctx


@pytest.mark.parametrize("kernel", ["", "tc"])
def test_one_workspace_serves_calls_of_different_shapes(kernel, monkeypatch):
    if kernel:
        monkeypatch.setenv("PKV_ATTN_KERNEL", kernel)
    BS = 16
    shapes = [(4, 32, 1, [3000, 17, 5000, 800]),          # few long segments of a 32-head group
              (64, 8, 8, [700 + 37 * i for i in range(64)]),   # many segments, one head each
              (3, 32, 8, [9000, 1, 4000]),
              (4, 32, 1, [3000, 17, 5000, 800])]
    need = max(pkv.decode_workspace_bytes(B, n_h, n_kv, 128, BS) for B, n_h, n_kv, _ in shapes)
    ws = torch.full((need,), 0xFF, dtype=torch.uint8, device=DEV)      # contents on entry do not matter
    for i, (B, n_h, n_kv, ctx) in enumerate(shapes):
        q, kp, vp, bt, ctx = _case(B, n_h, n_kv, ctx, BS, seed=10 + i)
        ref = oracle.paged_decode_attention(f64(q), f64(kp), f64(vp), bt, ctx, 1 / math.sqrt(128), BS)
        for od in (torch.bfloat16, torch.float32):
            err = err_flag()
            out = torch.full(q.shape, float("nan"), dtype=od, device=DEV)
            pkv.paged_decode_attn(q.to(DEV), kp.to(DEV), vp.to(DEV), torch.as_tensor(bt, device=DEV),
                                  torch.as_tensor(ctx, device=DEV), 1 / math.sqrt(128), out=out, workspace=ws,
                                  err=err)
            torch.cuda.synchronize()
            assert int(err.item()) == 0
            check_attention(out, ref, f"shape {i} {od}")


@pytest.mark.parametrize("kernel", ["", "tc"])
def test_a_segment_spread_over_hundreds_of_pieces(kernel, monkeypatch):
    if kernel:
        monkeypatch.setenv("PKV_ATTN_KERNEL", kernel)
    # one 32-head group over 40 000 tokens: the line of 2500 blocks is cut into as many
    # pieces as the grid has CTAs, every one holding part of the same segment
    BS = 16
    q, kp, vp, bt, ctx = _case(1, 32, 1, [40000], BS, seed=3)
    ref = oracle.paged_decode_attention(f64(q), f64(kp), f64(vp), bt, ctx, 0.1, BS)
    ws = torch.full((pkv.decode_workspace_bytes(1, 32, 1, 128, BS),), 0xFF, dtype=torch.uint8, device=DEV)
    outs = []
    for _ in range(2):
        err = err_flag()
        out = torch.full(q.shape, float("nan"), dtype=torch.float32, device=DEV)
        pkv.paged_decode_attn(q.to(DEV), kp.to(DEV), vp.to(DEV), torch.as_tensor(bt, device=DEV),
                              torch.as_tensor(ctx, device=DEV), 0.1, out=out, workspace=ws, err=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        check_attention(out, ref, f"40k tokens {kernel}")
        outs.append(out)
    assert torch.equal(outs[0], outs[1])


@pytest.mark.parametrize("D", [64, 128])
def test_long_segment_merges_alike_in_narrow_and_wide_reduce(D):
    # The split-reduce takes one CTA per row when segments are few, part of a warp per row
    # when they are many: the same 40 000-token sequence alone (8 segments, the grid's pieces
    # shared among them) and ahead of 199 short ones (1600 segments, more than the grid has
    # pieces; 6400 rows, more than one wave of warp-per-row CTAs, so half a warp per row)
    # goes through the two shapes, each compared with the oracle, in fp32 and bf16 output.
    BS, n_h, n_kv = 16, 32, 8
    scale = 1 / math.sqrt(D)
    q, kp, vp, bt, ctx = _case(200, n_h, n_kv, [40000] + [33 + 5 * i for i in range(199)], BS, seed=21, D=D)
    ref = oracle.paged_decode_attention(f64(q), f64(kp), f64(vp), bt, ctx, scale, BS)
    ws = torch.full((pkv.decode_workspace_bytes(200, n_h, n_kv, D, BS),), 0xFF, dtype=torch.uint8,
                    device=DEV)
    for B in (1, 200):
        for od in (torch.float32, torch.bfloat16):
            err = err_flag()
            out = torch.full((B, n_h, D), float("nan"), dtype=od, device=DEV)
            pkv.paged_decode_attn(q[:B].to(DEV), kp.to(DEV), vp.to(DEV), torch.as_tensor(bt[:B], device=DEV),
                                  torch.as_tensor(ctx[:B], device=DEV), scale, out=out, workspace=ws, err=err)
            torch.cuda.synchronize()
            assert int(err.item()) == 0
            check_attention(out, ref[:B], f"batch {B} D {D} {od}")
