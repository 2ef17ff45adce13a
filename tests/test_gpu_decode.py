"""Paged decode attention (bf16 cache) on the GPU against the fp64 oracle."""
import math

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_175_gb300 as pkv
import workloads
from gpu_common import DEV, check_attention, compact, f64, run_attention

pytestmark = pytest.mark.gpu


def _random_case(D, BS, n_h, n_kv, ctx, seed, pool_extra=5):
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
    kp = torch.randn(num_blocks, n_kv, BS, D, generator=g).to(torch.bfloat16)
    vp = torch.randn(num_blocks, n_kv, BS, D, generator=g).to(torch.bfloat16)
    q = torch.randn(len(ctx), n_h, D, generator=g).to(torch.bfloat16)
    return q, kp, vp, bt, ctx


@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
def test_tiny_workload(out_dtype):
    w = workloads.make("tiny", 0)
    kp, vp = workloads.pools_bf16(w, 0)
    q = workloads.queries(w, 0)
    ref = oracle.paged_decode_attention(f64(q), f64(kp), f64(vp), w.block_tables, w.context_lens, w.scale,
                                        w.block_size)
    out = run_attention(q.to(DEV), kp.to(DEV), vp.to(DEV), w.block_tables, w.context_lens, w.scale, out_dtype)
    check_attention(out, ref, f"tiny {out_dtype}")


SHAPES = [(8, 8), (8, 2), (32, 8), (32, 1), (64, 1), (48, 1), (16, 1), (6, 3)]


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("BS", [16, 32, 64])
@pytest.mark.parametrize("heads", SHAPES, ids=[f"{a}q{b}kv" for a, b in SHAPES])
def test_shape_sweep(D, BS, heads):
    n_h, n_kv = heads
    ctx = [0, 1, BS - 1, BS + 1, 3 * BS + 7, 2 * BS]
    q, kp, vp, bt, ctx = _random_case(D, BS, n_h, n_kv, ctx, seed=D * 1000 + BS * 10 + n_h)
    ref = oracle.paged_decode_attention(f64(q), f64(kp), f64(vp), bt, ctx, 1 / math.sqrt(D), BS)
    for od in (torch.bfloat16, torch.float32):
        out = run_attention(q.to(DEV), kp.to(DEV), vp.to(DEV), bt, ctx, 1 / math.sqrt(D), od)
        check_attention(out, ref, f"D{D} BS{BS} {n_h}/{n_kv} {od}")
        assert not f64(out)[0].any()                     # context length 0 -> zero row


def test_long_single_sequence_and_many_short():
    # one long segment cut across many pieces, plus many one-block sequences (whole in a piece)
    ctx = [20000] + [3] * 300 + [17, 0, 129]
    q, kp, vp, bt, ctx = _random_case(128, 16, 32, 8, ctx, seed=11)
    ref = oracle.paged_decode_attention(f64(q), f64(kp), f64(vp), bt, ctx, 0.0883883, 16)
    out = run_attention(q.to(DEV), kp.to(DEV), vp.to(DEV), bt, ctx, 0.0883883, torch.float32)
    check_attention(out, ref, "long+short f32")


def test_block_permutation_and_identity_table_are_bitwise_identical():
    q, kp, vp, bt, ctx = _random_case(128, 16, 32, 8, [700, 33, 1, 260], seed=3, pool_extra=40)
    a = run_attention(q.to(DEV), kp.to(DEV), vp.to(DEV), bt, ctx, 0.1)
    perm = np.random.default_rng(9).permutation(kp.shape[0])
    inv = np.argsort(perm)
    bt2 = np.where(bt >= 0, inv[np.maximum(bt, 0)], -1).astype(np.int32)
    b = run_attention(q.to(DEV), kp[perm].to(DEV), vp[perm].to(DEV), bt2, ctx, 0.1)
    assert torch.equal(a, b)
    # identity layout: each sequence's blocks stored contiguously in logical order
    nbs = [-(-int(c) // 16) for c in ctx]
    order = np.concatenate([bt[s, :n] for s, n in enumerate(nbs)])
    bt3 = np.full_like(bt, -1)
    cur = 0
    for s, n in enumerate(nbs):
        bt3[s, :n] = np.arange(cur, cur + n)
        cur += n
    c = run_attention(q.to(DEV), kp[order].contiguous().to(DEV), vp[order].contiguous().to(DEV), bt3, ctx, 0.1)
    assert torch.equal(a, c)


def test_gqa_matches_replicated_mha_on_gpu():
    q, kp, vp, bt, ctx = _random_case(128, 16, 32, 8, [300, 77, 1000], seed=5)
    a = run_attention(q.to(DEV), kp.to(DEV), vp.to(DEV), bt, ctx, 0.1, torch.float32)
    kr = kp.repeat_interleave(4, dim=1).contiguous()
    vr = vp.repeat_interleave(4, dim=1).contiguous()
    b = run_attention(q.to(DEV), kr.to(DEV), vr.to(DEV), bt, ctx, 0.1, torch.float32)
    assert torch.allclose(a, b, rtol=0, atol=2e-5)


def test_special_values():
    q, kp, vp, bt, ctx = _random_case(128, 16, 8, 2, [5, 40, 1], seed=8)
    ones = torch.ones_like(vp)
    out = run_attention(q.to(DEV), kp.to(DEV), ones.to(DEV), bt, ctx, 0.1)
    assert torch.equal(out, torch.ones_like(out))            # V == 1 gives exactly 1
    out = run_attention(torch.zeros_like(q).to(DEV), kp.to(DEV), vp.to(DEV), bt, ctx, 0.1, torch.float32)
    ref = oracle.paged_decode_attention(np.zeros(q.shape), f64(kp), f64(vp), bt, ctx, 0.1, 16)
    check_attention(out, ref, "q=0 (mean of V)")


def test_stale_values_past_the_context_do_not_leak():
    # rows past ctx in the last block hold inf / nan: they must not reach the output
    q, kp, vp, bt, ctx = _random_case(64, 16, 8, 2, [5, 21], seed=12)
    kp2, vp2 = kp.clone(), vp.clone()
    for s, c in enumerate(ctx):
        last = bt[s, (c - 1) // 16]
        kp2[last, :, c % 16:] = float("nan")
        vp2[last, :, c % 16:] = float("inf")
    ref = oracle.paged_decode_attention(f64(q), f64(kp), f64(vp), bt, ctx, 0.125, 16)
    out = run_attention(q.to(DEV), kp2.to(DEV), vp2.to(DEV), bt, ctx, 0.125, torch.float32)
    check_attention(out, ref, "stale rows")


def test_bad_block_id_sets_flag_and_is_skipped():
    q, kp, vp, bt, ctx = _random_case(128, 16, 8, 2, [40, 40], seed=13)
    bt_bad = bt.copy()
    bt_bad[1, 1] = kp.shape[0] + 7                         # out of range
    out = run_attention(q.to(DEV), kp.to(DEV), vp.to(DEV), bt_bad, ctx, 0.1, torch.float32,
                        expect_err=pkv.DEV_BAD_BLOCK)
    ref = oracle.paged_decode_attention(f64(q), f64(kp), f64(vp), bt, ctx, 0.1, 16)
    check_attention(out[:1], ref[:1], "untouched sequence")
    assert torch.isfinite(out).all()


def test_context_beyond_table_is_clamped_and_flagged():
    q, kp, vp, bt, ctx = _random_case(64, 16, 8, 2, [32, 20], seed=14)
    bad_ctx = np.array([32, 10 ** 6], dtype=np.int32)
    run_attention(q.to(DEV), kp.to(DEV), vp.to(DEV), bt, bad_ctx, 0.1, expect_err=pkv.DEV_BAD_CTX)


FULL = ["llama3_8b", "llama2_70b_prefix", "mqa_bs16", "mqa_bs32", "mha_bs16", "mha_bs32"]


@pytest.mark.parametrize("name", FULL)
def test_full_size_step_sampled(name):
    """The benchmark's decode step (append, then attend) at full size; sampled rows vs the oracle."""
    w = workloads.make(name, 0)
    kp, vp = workloads.pools_bf16(w, 0, DEV)
    q = workloads.queries(w, 0, DEV)
    kn, vn = workloads.new_tokens(w, 0, DEV)
    slots = workloads.decode_slots(w)
    order = np.argsort(w.context_lens)
    seqs = sorted({int(order[0]), int(order[-1]), 0, 1, w.batch // 2, w.batch - 1})
    phys, cbt, cctx = compact(w.block_tables, w.context_lens, seqs, w.block_size)
    idx = torch.as_tensor(phys, device=DEV)
    k_before, v_before = f64(kp[idx]), f64(vp[idx])            # the cache before this step's append
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    pkv.kv_append(kn, vn, torch.as_tensor(slots, device=DEV), kp, vp, err=err)
    bt, ctx = torch.as_tensor(w.block_tables, device=DEV), torch.as_tensor(w.context_lens, device=DEV)
    out = pkv.paged_decode_attn(q, kp, vp, bt, ctx, w.scale, err=err)
    out32 = pkv.paged_decode_attn(q, kp, vp, bt, ctx, w.scale, out_dtype=torch.float32, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    # oracle: its own append on the compact copy, then attention
    remap = {int(p): i for i, p in enumerate(phys)}
    cslots = np.array([remap[int(slots[s]) // w.block_size] * w.block_size + int(slots[s]) % w.block_size
                       for s in seqs], dtype=np.int64)
    k_after, v_after = oracle.kv_append(k_before, v_before, f64(kn[seqs]), f64(vn[seqs]), cslots, w.block_size)
    ref = oracle.paged_decode_attention(f64(q[seqs]), k_after, v_after, cbt, cctx, w.scale, w.block_size)
    check_attention(out32[seqs], ref, name)
    check_attention(out[seqs], ref, name)
