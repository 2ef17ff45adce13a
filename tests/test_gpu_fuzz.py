"""Seeded random shapes against the fp64 oracle: head layouts, block sizes, context mixes
(including lengths on and just off block boundaries) and attention windows, for the bf16
and the INT4 cache.  The partition then cuts segments at many offsets, so stages of one
and of two blocks, pieces that start mid-segment and windows that start inside a stage all
occur; every case is compared element by element with fp32 output."""
import math

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_175_gb300 as pkv
from gpu_common import BAR_INT4_F32_MAXABS, BAR_INT4_F32_RELL2, DEV, check_attention, err_flag, f64
from test_gpu_decode import _random_case
from test_gpu_int4 import _append_both, _history, _tables

pytestmark = pytest.mark.gpu

HEADS = [(8, 8), (8, 1), (8, 2), (32, 4), (32, 1), (16, 2), (6, 3)]


def _contexts(rng, BS):
    batch = int(rng.integers(1, 25))
    ctx = rng.integers(1, 700, size=batch)
    edge = rng.random(batch) < 0.3                         # on, and one past, a block boundary
    ctx[edge] = (ctx[edge] // BS) * BS + rng.integers(0, 2, size=int(edge.sum()))
    return np.maximum(ctx, 1).astype(np.int32)


@pytest.mark.parametrize("seed", range(16))
def test_bf16_random_shapes(seed):
    rng = np.random.default_rng(1000 + seed)
    D = int(rng.choice([64, 128]))
    BS = int(rng.choice([16, 32, 64]))
    n_h, n_kv = HEADS[int(rng.integers(len(HEADS)))]
    ctx = _contexts(rng, BS)
    window = 0 if seed % 3 == 0 else int(rng.integers(1, 300))
    q, kp, vp, bt, ctx = _random_case(D, BS, n_h, n_kv, ctx, seed=2000 + seed)
    scale = 1 / math.sqrt(D)
    ref = oracle.paged_decode_attention(f64(q), f64(kp), f64(vp), bt, ctx, scale, BS, window=window)
    err = err_flag()
    out = pkv.paged_decode_attn_window(q.to(DEV), kp.to(DEV), vp.to(DEV), torch.as_tensor(bt, device=DEV),
                                       torch.as_tensor(ctx, device=DEV), scale, window, out_dtype=torch.float32,
                                       err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    check_attention(out, ref, f"bf16 D{D} BS{BS} {n_h}/{n_kv} window {window} batch {len(ctx)}")


@pytest.mark.parametrize("seed", range(10))
def test_int4_random_shapes(seed):
    rng = np.random.default_rng(3000 + seed)
    D = int(rng.choice([64, 128]))
    BS = int(rng.choice([16, 16, 32, 64]))
    n_h, n_kv = HEADS[int(rng.integers(len(HEADS)))]
    ctx = _contexts(rng, BS)
    window = 0 if seed % 3 == 0 else int(rng.integers(1, 300))
    bt, num_blocks = _tables(ctx, BS, rng)
    ks, vs = _history(ctx, n_kv, D, seed=4000 + seed)
    cache = pkv.alloc_int4_cache(num_blocks, n_kv, BS, D, len(ctx), DEV)
    ref = oracle.Int4Cache(num_blocks, n_kv, BS, D, len(ctx))
    sl = np.concatenate([bt[s, np.arange(c) // BS].astype(np.int64) * BS + np.arange(c) % BS
                         for s, c in enumerate(ctx)])
    tl = np.concatenate([np.full(c, s) for s, c in enumerate(ctx)])
    _append_both(cache, ref, torch.cat(ks), torch.cat(vs), sl, tl)
    q = torch.randn(len(ctx), n_h, D, generator=torch.Generator().manual_seed(5000 + seed)).to(torch.bfloat16)
    scale = 1 / math.sqrt(D)
    refo = oracle.paged_decode_attention_int4(f64(q), ref, bt, ctx, scale, window=window)
    err = err_flag()
    out = pkv.paged_decode_attn_int4_window(q.to(DEV), cache, torch.as_tensor(bt, device=DEV),
                                            torch.as_tensor(ctx, device=DEV), scale, window,
                                            out_dtype=torch.float32, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    check_attention(out, refo, f"int4 D{D} BS{BS} {n_h}/{n_kv} window {window} batch {len(ctx)}",
                    f32_bars=(BAR_INT4_F32_MAXABS, BAR_INT4_F32_RELL2))
