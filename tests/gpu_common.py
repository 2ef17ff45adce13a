"""Helpers shared by the GPU parity tests (not a test module)."""
import numpy as np
import torch

import oracle
import paged_kv_cache_175_gb300 as pkv

DEV = "cuda"

# Bars.  bf16 output: the stated bound against the fp64 oracle, and against the
# oracle's own bf16 rounding of its result (at most one bf16 ulp apart, almost all
# identical).  fp32 output: the kernel's arithmetic alone (tight).
BAR_BF16_MAXABS, BAR_BF16_RELL2 = 1e-2, 2e-3
BAR_F32_MAXABS, BAR_F32_RELL2 = 5e-4, 5e-5
BAR_INT4_F32_MAXABS, BAR_INT4_F32_RELL2 = 2e-3, 5e-4


def f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def rel_l2(a, b):
    nb = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / nb) if nb > 0 else float(np.linalg.norm(a - b))


def bf16_ulp(x):
    x = np.abs(np.asarray(x, dtype=np.float64))
    e = np.floor(np.log2(np.maximum(x, 2.0 ** -126)))
    return 2.0 ** (e - 7)


def attention_stats(got: np.ndarray, ref: np.ndarray) -> dict:
    """Errors of a bf16 / fp32 output against the fp64 result.  `ulps_max` counts bf16 ulps
    from the oracle's own rounding, with an absolute floor of 1e-5 * max|ref| (an output
    near zero is a cancellation: its fp32 error is absolute, not relative)."""
    rb = oracle.round_bf16(ref)
    d = np.abs(got - rb)
    floor = 1e-5 * float(np.abs(ref).max())
    return {"maxabs": float(np.abs(got - ref).max()), "rel_l2": rel_l2(got, ref),
            "ulps_max": float((np.maximum(d - floor, 0) / bf16_ulp(rb)).max()), "exact": float(np.mean(d == 0))}


def check_attention(out: torch.Tensor, ref: np.ndarray, what: str, f32_bars=(BAR_F32_MAXABS, BAR_F32_RELL2),
                    min_exact=0.99):
    """Compare a GPU attention output with the fp64 oracle result."""
    got = f64(out)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    assert np.isfinite(got).all(), what
    st = attention_stats(got, ref)
    msg = (what, str(out.dtype), st)
    if out.dtype == torch.float32:
        assert st["maxabs"] <= f32_bars[0] and st["rel_l2"] <= f32_bars[1], msg
        return
    assert st["maxabs"] <= BAR_BF16_MAXABS and st["rel_l2"] <= BAR_BF16_RELL2, msg
    assert st["ulps_max"] <= 1.0001, msg
    assert st["exact"] >= min_exact, msg


def compact(block_tables: np.ndarray, context_lens: np.ndarray, seqs, block_size: int):
    """Physical blocks used by `seqs`, and their tables re-indexed into a compact pool.

    Returns (phys_ids int64 [n], tables int32 [len(seqs)][max_blocks], ctx int32 [len(seqs)]).
    Paging is a pure layout change (pinned in the oracle tests), so attention over the
    compact pool equals attention over the full one.
    """
    used = []
    for s in seqs:
        nb = -(-int(context_lens[s]) // block_size)
        used.extend(block_tables[s, :nb].tolist())
    phys = np.unique(np.array(used, dtype=np.int64))
    remap = {int(p): i for i, p in enumerate(phys)}
    mb = max(1, max(-(-int(context_lens[s]) // block_size) for s in seqs))
    bt = np.full((len(seqs), mb), -1, dtype=np.int32)
    for r, s in enumerate(seqs):
        nb = -(-int(context_lens[s]) // block_size)
        bt[r, :nb] = [remap[int(p)] for p in block_tables[s, :nb]]
    return phys, bt, np.asarray([context_lens[s] for s in seqs], dtype=np.int32)


def err_flag():
    return torch.zeros(1, dtype=torch.int32, device=DEV)


def run_attention(q, k_pool, v_pool, bt, ctx, scale, out_dtype=torch.bfloat16, expect_err=0):
    err = err_flag()
    out = pkv.paged_decode_attn(q, k_pool, v_pool, torch.as_tensor(bt, device=DEV),
                                torch.as_tensor(ctx, device=DEV), scale, out_dtype=out_dtype, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == expect_err, int(err.item())
    return out
