"""INT4 quantize-on-append (byte-exact) and INT4 decode attention on the GPU vs the oracle."""
import math

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_175_gb300 as pkv
import workloads
from gpu_common import (BAR_INT4_F32_MAXABS, BAR_INT4_F32_RELL2, DEV, check_attention, compact, err_flag,
                        f64)

pytestmark = pytest.mark.gpu


def _tables(ctx, BS, rng, extra=3):
    nbs = [-(-int(c) // BS) for c in ctx]
    num_blocks = sum(nbs) + extra
    perm = rng.permutation(num_blocks).astype(np.int32)
    bt = np.full((len(ctx), max(1, max(nbs))), -1, dtype=np.int32)
    cur = 0
    for s, n in enumerate(nbs):
        bt[s, :n] = perm[cur:cur + n]
        cur += n
    return bt, num_blocks


def _history(ctx, n_kv, D, seed, outliers=True):
    g = torch.Generator().manual_seed(seed)
    ks, vs = [], []
    for c in ctx:
        k = torch.randn(int(c), n_kv, D, generator=g)
        if outliers:
            k[:, :, [3, D // 2 + 1]] *= 10.0
        ks.append(k.to(torch.bfloat16))
        vs.append(torch.randn(int(c), n_kv, D, generator=g).to(torch.bfloat16))
    return ks, vs


def _compare_state(cache: pkv.Int4CacheTensors, ref: oracle.Int4Cache, blocks, rows):
    assert np.array_equal(cache.k_codes.cpu().numpy()[blocks], ref.k_codes[blocks])
    assert np.array_equal(cache.v_codes.cpu().numpy()[blocks], ref.v_codes[blocks])
    assert cache.k_meta.cpu().numpy()[blocks].tobytes() == ref.k_meta[blocks].tobytes()
    assert cache.v_meta.cpu().numpy()[blocks].tobytes() == ref.v_meta[blocks].tobytes()
    assert np.array_equal(f64(cache.k_tail)[rows], ref.k_tail[rows])


def _append_both(cache, ref, k, v, slots, tails):
    err = err_flag()
    pkv.kv_quant_append_int4(k.to(DEV), v.to(DEV), torch.as_tensor(slots, device=DEV),
                             torch.as_tensor(tails, dtype=torch.int32, device=DEV), cache, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ref.append(f64(k), f64(v), slots, tails)


@pytest.mark.parametrize("D,BS", [(128, 16), (64, 16), (128, 64), (128, 32)])
def test_bulk_then_streaming_append_and_attention(D, BS):
    rng = np.random.default_rng(D + BS)
    n_kv, n_h = 2, 8
    final = np.array([5, BS, 3 * BS + 7, 2 * BS - 1, 1], dtype=np.int32)
    prefill = np.array([3, BS - 2, 2 * BS + 1, BS, 0], dtype=np.int32)
    bt, num_blocks = _tables(final, BS, rng)
    ks, vs = _history(final, n_kv, D, seed=D * BS)
    cache = pkv.alloc_int4_cache(num_blocks, n_kv, BS, D, len(final), DEV)
    ref = oracle.Int4Cache(num_blocks, n_kv, BS, D, len(final))
    # prefill: every sequence's first tokens in one call (consecutive per sequence)
    kk, vv, sl, tl = [], [], [], []
    for s, c in enumerate(prefill):
        pos = np.arange(c)
        kk.append(ks[s][:c]); vv.append(vs[s][:c])
        sl.append(bt[s, pos // BS].astype(np.int64) * BS + pos % BS); tl.append(np.full(c, s))
    _append_both(cache, ref, torch.cat(kk), torch.cat(vv), np.concatenate(sl), np.concatenate(tl))
    allb = np.arange(num_blocks)
    _compare_state(cache, ref, allb, np.arange(len(final)))
    # then decode steps: one token per unfinished sequence per call
    for t in range(int((final - prefill).max())):
        live = [s for s in range(len(final)) if prefill[s] + t < final[s]]
        pos = np.array([prefill[s] + t for s in live])
        slots = np.array([bt[s, p // BS] * BS + p % BS for s, p in zip(live, pos)], dtype=np.int64)
        _append_both(cache, ref, torch.stack([ks[s][p] for s, p in zip(live, pos)]),
                     torch.stack([vs[s][p] for s, p in zip(live, pos)]), slots, np.array(live))
    _compare_state(cache, ref, allb, np.arange(len(final)))
    # attention on each side's own (identical) state
    g = torch.Generator().manual_seed(3)
    q = torch.randn(len(final), n_h, D, generator=g).to(torch.bfloat16)
    refo = oracle.paged_decode_attention_int4(f64(q), ref, bt, final, 1 / math.sqrt(D))
    for od in (torch.bfloat16, torch.float32):
        err = err_flag()
        out = pkv.paged_decode_attn_int4(q.to(DEV), cache, torch.as_tensor(bt, device=DEV),
                                         torch.as_tensor(final, device=DEV), 1 / math.sqrt(D), out_dtype=od,
                                         err=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        check_attention(out, refo, f"int4 D{D} BS{BS} {od}", f32_bars=(BAR_INT4_F32_MAXABS, BAR_INT4_F32_RELL2),
                        min_exact=0.95)


@pytest.mark.parametrize("heads", [(8, 8), (32, 1), (64, 2)])
def test_int4_group_sizes(heads):
    n_h, n_kv = heads
    D, BS = 128, 16
    rng = np.random.default_rng(n_h)
    ctx = np.array([40, 16, 100], dtype=np.int32)
    bt, num_blocks = _tables(ctx, BS, rng)
    ks, vs = _history(ctx, n_kv, D, seed=n_h)
    cache = pkv.alloc_int4_cache(num_blocks, n_kv, BS, D, len(ctx), DEV)
    ref = oracle.Int4Cache(num_blocks, n_kv, BS, D, len(ctx))
    sl = np.concatenate([bt[s, np.arange(c) // BS].astype(np.int64) * BS + np.arange(c) % BS
                         for s, c in enumerate(ctx)])
    tl = np.concatenate([np.full(c, s) for s, c in enumerate(ctx)])
    _append_both(cache, ref, torch.cat(ks), torch.cat(vs), sl, tl)
    q = torch.randn(len(ctx), n_h, D, generator=torch.Generator().manual_seed(1)).to(torch.bfloat16)
    refo = oracle.paged_decode_attention_int4(f64(q), ref, bt, ctx, 0.088)
    out = pkv.paged_decode_attn_int4(q.to(DEV), cache, torch.as_tensor(bt, device=DEV),
                                     torch.as_tensor(ctx, device=DEV), 0.088, out_dtype=torch.float32)
    torch.cuda.synchronize()
    check_attention(out, refo, f"int4 {n_h}/{n_kv}", f32_bars=(BAR_INT4_F32_MAXABS, BAR_INT4_F32_RELL2))


def test_long_segment_through_both_reduce_shapes():
    # One 20 000-token INT4 sequence (8 kv heads) alone -- its segments spread over about 150
    # pieces each, merged by the one-CTA-per-row reduce -- and ahead of 199 short ones (6400
    # rows: half a warp per row), both against the oracle.
    D, BS, n_kv, n_h = 128, 16, 8, 32
    ctx = np.array([20000] + [33 + 5 * i for i in range(199)], dtype=np.int32)
    rng = np.random.default_rng(11)
    bt, num_blocks = _tables(ctx, BS, rng)
    ks, vs = _history(ctx, n_kv, D, seed=12)
    cache = pkv.alloc_int4_cache(num_blocks, n_kv, BS, D, len(ctx), DEV)
    ref = oracle.Int4Cache(num_blocks, n_kv, BS, D, len(ctx))
    sl = np.concatenate([bt[s, np.arange(c) // BS].astype(np.int64) * BS + np.arange(c) % BS
                         for s, c in enumerate(ctx)])
    tl = np.concatenate([np.full(c, s) for s, c in enumerate(ctx)])
    _append_both(cache, ref, torch.cat(ks), torch.cat(vs), sl, tl)
    q = torch.randn(len(ctx), n_h, D, generator=torch.Generator().manual_seed(13)).to(torch.bfloat16)
    scale = 1 / math.sqrt(D)
    refo = oracle.paged_decode_attention_int4(f64(q), ref, bt, ctx, scale)
    for B in (1, len(ctx)):
        err = err_flag()
        out = pkv.paged_decode_attn_int4(q[:B].to(DEV), cache, torch.as_tensor(bt[:B], device=DEV),
                                         torch.as_tensor(ctx[:B], device=DEV), scale, out_dtype=torch.float32,
                                         err=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        check_attention(out, refo[:B], f"int4 long segment, batch {B}",
                        f32_bars=(BAR_INT4_F32_MAXABS, BAR_INT4_F32_RELL2))


def test_bad_tail_row_flagged():
    cache = pkv.alloc_int4_cache(4, 1, 16, 64, 2, DEV)
    k = torch.ones(1, 1, 64, dtype=torch.bfloat16, device=DEV)
    err = err_flag()
    pkv.kv_quant_append_int4(k, k, torch.tensor([3], device=DEV), torch.tensor([5], dtype=torch.int32, device=DEV),
                             cache, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == pkv.DEV_BAD_SLOT
    assert not cache.v_codes.any() and not cache.k_tail.any()


@pytest.mark.parametrize("name", ["int4_long", "int4_long_bs64"])
def test_full_size_sampled(name):
    """The long-context INT4 workload at full size: bulk quantize-on-append of every
    sequence's history, then one decode step; one sampled sequence against the oracle."""
    w = workloads.make(name, 0)
    BS = w.block_size
    cache = pkv.alloc_int4_cache(w.num_blocks, w.n_kv, BS, w.head_dim, w.batch, DEV)
    hist = [workloads.history_kv(w, s, 0, DEV) for s in range(w.batch)]
    k_all = torch.cat([h[0] for h in hist])
    v_all = torch.cat([h[1] for h in hist])
    slots = np.concatenate([workloads.history_slots(w, s) for s in range(w.batch)])
    tails = np.concatenate([np.full(int(c), s, np.int32) for s, c in enumerate(w.context_lens)])
    err = err_flag()
    pkv.kv_quant_append_int4(k_all, v_all, torch.as_tensor(slots, device=DEV), torch.as_tensor(tails, device=DEV),
                             cache, err=err)
    q = workloads.queries(w, 0, DEV)
    out = pkv.paged_decode_attn_int4(q, cache, torch.as_tensor(w.block_tables, device=DEV),
                                     torch.as_tensor(w.context_lens, device=DEV), w.scale, err=err)
    out32 = pkv.paged_decode_attn_int4(q, cache, torch.as_tensor(w.block_tables, device=DEV),
                                       torch.as_tensor(w.context_lens, device=DEV), w.scale,
                                       out_dtype=torch.float32, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    # the shortest, the median and the longest history: the longest is cut across the most
    # pieces (every split merge), and each ends in an unfinished block read from the tail
    order = np.argsort(w.context_lens, kind="stable")
    for s in (int(order[0]), int(order[len(order) // 2]), int(order[-1])):
        phys, cbt, cctx = compact(w.block_tables, w.context_lens, [s], BS)
        ref = oracle.Int4Cache(len(phys), w.n_kv, BS, w.head_dim, 1)
        pos = np.arange(int(w.context_lens[s]))
        ref.append(f64(hist[s][0]), f64(hist[s][1]), cbt[0, pos // BS].astype(np.int64) * BS + pos % BS,
                   np.zeros(len(pos), np.int32))
        idx = torch.as_tensor(phys, device=DEV)
        assert np.array_equal(cache.k_codes[idx].cpu().numpy(), ref.k_codes)
        assert np.array_equal(cache.v_codes[idx].cpu().numpy(), ref.v_codes)
        assert cache.k_meta[idx].cpu().numpy().tobytes() == ref.k_meta.tobytes()
        assert cache.v_meta[idx].cpu().numpy().tobytes() == ref.v_meta.tobytes()
        refo = oracle.paged_decode_attention_int4(f64(q[s:s + 1]), ref, cbt, cctx, w.scale)
        check_attention(out[s:s + 1], refo, f"{name} seq {s} ctx {int(w.context_lens[s])}", min_exact=0.95)
        check_attention(out32[s:s + 1], refo, f"{name} seq {s} fp32",
                        f32_bars=(BAR_INT4_F32_MAXABS, BAR_INT4_F32_RELL2))


@pytest.mark.parametrize("D,BS", [(128, 16), (64, 32)])
def test_codes_on_exact_ties_round_half_to_even(D, BS):
    # Every group spans [0, 7.5] exactly, so s = 0.5 and min = 0 are exact in fp16 and every
    # other value 0.25 + 0.5 k sits exactly on a tie (quotient k + 0.5): the codes must be the
    # oracle's round-half-to-even of the exact quotient, with ties mixed among ordinary values
    rng = np.random.default_rng(D + BS)
    n_kv = 2
    def grid(shape):
        x = 0.25 + 0.5 * rng.integers(0, 15, size=shape)
        plain = rng.random(shape) < 0.3
        x[plain] = 0.5 * rng.integers(0, 16, size=plain.sum())     # exact codes, no tie
        return x
    k = grid((BS, n_kv, D))
    k[0], k[1] = 0.0, 7.5                                  # each channel's K range over the block
    v = grid((BS, n_kv, D))
    v[:, :, 0], v[:, :, 1] = 0.0, 7.5                      # each token's V range
    k, v = torch.tensor(k).to(torch.bfloat16), torch.tensor(v).to(torch.bfloat16)
    assert torch.equal(k.double(), torch.tensor(k.double().numpy()))   # all values exact in bf16
    num_blocks = 3
    cache = pkv.alloc_int4_cache(num_blocks, n_kv, BS, D, 1, DEV)
    ref = oracle.Int4Cache(num_blocks, n_kv, BS, D, 1)
    slots = np.arange(BS, dtype=np.int64) + BS                        # block 1, all rows
    _append_both(cache, ref, k, v, slots, np.zeros(BS, np.int32))
    _compare_state(cache, ref, [1], [0])
