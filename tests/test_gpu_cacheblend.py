"""CacheBlend's model-free steps on the GPU against the oracle: KV deviation (float tolerance
against fp64), selection (bit-exact on the same float32 values), fuse (bit-exact)."""
import numpy as np
import pytest
import torch

import paged_kv_cache_175_gb300 as pkv
import workloads
from oracle import cacheblend as cb
from gpu_common import DEV, err_flag, f64

pytestmark = pytest.mark.gpu


def _case(n_kv, d, bs, n, seed, N=None):
    g = torch.Generator().manual_seed(seed)
    N = N or (n // bs + 8)
    kp = torch.randn(N, n_kv, bs, d, generator=g).to(torch.bfloat16)
    vp = torch.randn(N, n_kv, bs, d, generator=g).to(torch.bfloat16)
    rng = np.random.default_rng(seed)
    slots = rng.permutation(N * bs)[:n].astype(np.int64)
    blk, row = slots // bs, slots % bs
    scale = torch.as_tensor(rng.exponential(0.3, size=(n, 1, 1)), dtype=torch.float32)
    kn = (kp[blk, :, row].float() + scale * torch.randn(n, n_kv, d, generator=g)).to(torch.bfloat16)
    vn = (vp[blk, :, row].float() + scale * torch.randn(n, n_kv, d, generator=g)).to(torch.bfloat16)
    return kp, vp, slots, kn, vn


@pytest.mark.parametrize("shape", [(1, 128), (8, 128), (32, 128), (2, 64)], ids=lambda s: f"{s[0]}kv{s[1]}")
@pytest.mark.parametrize("n", [1, 33, 1000])
def test_deviation_against_fp64(shape, n):
    n_kv, d = shape
    bs = 16
    kp, vp, slots, kn, vn = _case(n_kv, d, bs, n, seed=n_kv * 7 + n)
    ref = cb.kv_deviation(f64(kp), f64(vp), slots, f64(kn), f64(vn), bs)
    err = err_flag()
    got = pkv.kv_deviation(kp.to(DEV), vp.to(DEV), torch.as_tensor(slots, device=DEV), kn.to(DEV), vn.to(DEV),
                           err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    got = f64(got)
    # fp32 accumulation of squares of exact differences: relative error a few 1e-7 * sqrt(terms)
    assert np.all(np.abs(got - ref) <= 2e-5 * ref + 1e-6), float(np.max(np.abs(got - ref) / np.maximum(ref, 1e-9)))


def test_deviation_of_identical_rows_is_zero_and_bad_slot_flagged():
    kp, vp, slots, _, _ = _case(4, 128, 16, 50, seed=3)
    blk, row = slots // 16, slots % 16
    kn, vn = kp[blk, :, row].contiguous(), vp[blk, :, row].contiguous()
    err = err_flag()
    s = torch.as_tensor(slots, device=DEV)
    got = pkv.kv_deviation(kp.to(DEV), vp.to(DEV), s, kn.to(DEV), vn.to(DEV), err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0 and not got.any()
    s[5] = kp.shape[0] * 16
    got = pkv.kv_deviation(kp.to(DEV), vp.to(DEV), s, kn.to(DEV), vn.to(DEV), err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == pkv.DEV_BAD_SLOT and float(got[5]) == 0.0


@pytest.mark.parametrize("seed", range(4))
def test_selection_is_exact(seed):
    rng = np.random.default_rng(seed)
    lens = [0, 1, 5, 1023, 1024, 1025, 3000, 20000, 77]
    offs = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    dev = (np.round(rng.random(offs[-1]) * (64 if seed % 2 else 1e6)) / 8).astype(np.float32)   # ties when coarse
    counts = [0, 1, 7, 100, 1024, 154, 451, 3000, 200]                                        # k > n clamps
    got = pkv.select_top(torch.as_tensor(dev, device=DEV), offs, counts).cpu().numpy().tolist()
    want = cb.select_top_segments(dev.astype(np.float64), offs, [min(c, l) for c, l in zip(counts, lens)])
    assert got == want


def test_fuse_is_exact():
    kp, vp, _, _, _ = _case(8, 128, 16, 10, seed=5, N=40)
    rng = np.random.default_rng(6)
    kn = torch.randn(200, 8, 128).to(torch.bfloat16)
    vn = torch.randn(200, 8, 128).to(torch.bfloat16)
    rows = rng.choice(200, size=60, replace=False).astype(np.int32)
    row_slots = rng.permutation(40 * 16)[:200].astype(np.int64)          # a distinct slot per candidate row
    kd, vd = kp.to(DEV), vp.to(DEV)
    err = err_flag()
    pkv.kv_fuse(kn.to(DEV), vn.to(DEV), torch.as_tensor(row_slots, device=DEV), torch.as_tensor(rows, device=DEV),
                kd, vd, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    bits = lambda t: t.cpu().view(torch.int16).numpy()
    rk, rv = cb.fuse(bits(kp), bits(vp), bits(kn), bits(vn), rows, row_slots[rows], 16)
    assert np.array_equal(bits(kd), rk) and np.array_equal(bits(vd), rv)


@pytest.mark.parametrize("name", ["mqa_bs16", "mha_bs32"])
def test_full_size_layer_step(name):
    """One layer of CacheBlend on the 64 reused 512-token chunks of the workload: deviation
    of every chunk token against synthetic recomputed K/V, 15% of each chunk selected, the
    selected rows fused into the cache.  Deviation sampled against fp64, selection exact on
    the GPU's values, the fused rows hold the recomputed values and no other row changed."""
    w = workloads.make(name, 0)
    bs = w.block_size
    kp, vp = workloads.pools_bf16(w, 0, DEV)
    blocks = w.extra["rope_block_ids"].astype(np.int64)
    slots = (blocks[:, None] * bs + np.arange(bs)[None, :]).reshape(-1)          # 64 x 512 tokens
    n = len(slots)
    g = torch.Generator(device=DEV).manual_seed(9)
    blk = torch.as_tensor(slots // bs, device=DEV)
    row = torch.as_tensor(slots % bs, device=DEV)
    scale = torch.rand(n, 1, 1, generator=g, device=DEV) ** 3
    kn = (kp[blk, :, row].float() + scale * torch.randn(n, w.n_kv, w.head_dim, generator=g, device=DEV)).to(torch.bfloat16)
    vn = (vp[blk, :, row].float() + scale * torch.randn(n, w.n_kv, w.head_dim, generator=g, device=DEV)).to(torch.bfloat16)
    err = err_flag()
    s_d = torch.as_tensor(slots, device=DEV)
    dev = pkv.kv_deviation(kp, vp, s_d, kn, vn, err=err)
    offs = np.arange(0, n + 1, 512, dtype=np.int32)
    k = pkv.select_count(0.15, 512)
    sel = pkv.select_top(dev, offs, [k] * 64)
    k_before, v_before = kp.clone(), vp.clone()
    pkv.kv_fuse(kn, vn, s_d, sel, kp, vp, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0 and sel.numel() == 64 * k
    # deviation: sampled tokens against fp64
    idx = np.random.default_rng(1).choice(n, size=64, replace=False)
    kb = f64(k_before[blk[idx], :, row[idx]]).reshape(len(idx), 1, w.n_kv, w.head_dim).transpose(0, 2, 1, 3)
    vb = f64(v_before[blk[idx], :, row[idx]]).reshape(len(idx), 1, w.n_kv, w.head_dim).transpose(0, 2, 1, 3)
    ref = cb.kv_deviation(kb, vb, np.arange(len(idx)), f64(kn[idx]), f64(vn[idx]), 1)
    got = f64(dev)[idx]
    assert np.all(np.abs(got - ref) <= 2e-5 * ref + 1e-6)
    # selection: exact on the GPU's float32 values
    dv = dev.cpu().numpy()
    sel_np = sel.cpu().numpy()
    assert sel_np.tolist() == cb.select_top_segments(dv.astype(np.float64), offs, [k] * 64)
    # fuse: the selected rows now hold the recomputed rows; no other row changed
    sb, sr = blk[sel.long()], row[sel.long()]
    assert torch.equal(kp[sb, :, sr], kn[sel.long()]) and torch.equal(vp[sb, :, sr], vn[sel.long()])
    changed = (kp != k_before).flatten(3).any(-1) | (vp != v_before).flatten(3).any(-1)   # [blocks][kv][rows]
    mask = torch.zeros_like(changed)
    mask[sb, :, sr] = True
    assert not (changed & ~mask).any()
