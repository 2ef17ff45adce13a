"""Block copies between the GPU pools and page-locked host pools (offload / onload), and
the block manager driving a real paged cache through them, against the oracle."""
import math

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_175_gb300 as pkv
from gpu_common import DEV, check_attention, err_flag, f64

pytestmark = pytest.mark.gpu


def _pools(N, H, n_kv, bs, d, seed):
    g = torch.Generator().manual_seed(seed)
    kp = torch.randn(N, n_kv, bs, d, generator=g).to(torch.bfloat16)
    vp = torch.randn(N, n_kv, bs, d, generator=g).to(torch.bfloat16)
    kh = torch.randn(H, n_kv, bs, d, generator=g).to(torch.bfloat16).pin_memory()
    vh = torch.randn(H, n_kv, bs, d, generator=g).to(torch.bfloat16).pin_memory()
    return kp, vp, kh, vh


def _bits(t):
    return t.cpu().view(torch.int16).numpy()


@pytest.mark.parametrize("n_copies", [1, 7, 600, 2000])
def test_copy_blocks_equals_sequential_application(n_copies):
    N, H, n_kv, bs, d = 64, 48, 2, 16, 128
    kp, vp, kh, vh = _pools(N, H, n_kv, bs, d, n_copies)
    rng = np.random.default_rng(n_copies)
    # random copies with many dependencies (repeated blocks and slots in both roles)
    kinds = rng.integers(0, 2, size=n_copies)
    copies = np.stack([kinds, np.where(kinds == 0, rng.integers(0, N, n_copies), rng.integers(0, H, n_copies)),
                       np.where(kinds == 0, rng.integers(0, H, n_copies), rng.integers(0, N, n_copies))], 1)
    ref_k, ref_v, ref_kh, ref_vh = _bits(kp).copy(), _bits(vp).copy(), _bits(kh).copy(), _bits(vh).copy()
    oracle.apply_copies(copies, ref_k, ref_kh)
    oracle.apply_copies(copies, ref_v, ref_vh)
    kd, vd = kp.to(DEV), vp.to(DEV)
    pkv.copy_blocks(copies, kd, vd, kh, vh)
    torch.cuda.synchronize()
    assert np.array_equal(_bits(kd), ref_k) and np.array_equal(_bits(vd), ref_v)
    assert np.array_equal(_bits(kh), ref_kh) and np.array_equal(_bits(vh), ref_vh)


def test_copy_blocks_rejects_bad_input():
    kp, vp, kh, vh = _pools(4, 2, 1, 16, 64, 0)
    kd, vd = kp.to(DEV), vp.to(DEV)
    with pytest.raises(pkv.PkvError):
        pkv.copy_blocks([[0, 4, 0]], kd, vd, kh, vh)          # GPU block out of range
    with pytest.raises(pkv.PkvError):
        pkv.copy_blocks([[1, 2, 0]], kd, vd, kh, vh)          # host slot out of range
    with pytest.raises(pkv.PkvError):
        pkv.copy_blocks([[2, 0, 0]], kd, vd, kh, vh)          # unknown kind
    with pytest.raises(pkv.PkvError):
        pkv.copy_blocks([[0, 0, 0]], kd, vd, kh.clone(), vh)  # not page-locked


def _kv_of(token, pos, n_kv, d, table):
    """K / V rows of a token at a position: a fixed function of both (bf16)."""
    return table[token % len(table)] + 0.01 * (pos % 97)


def test_manager_drives_a_cache_through_offload_and_onload():
    """Requests over shared prefixes on a small pool with a host tier: prefill and decode
    writes go to the manager's slots, recorded copies are applied before each write, and at
    the end every running sequence's attention equals the oracle's over its own tokens."""
    N, H, n_kv, bs, d, n_h = 40, 24, 2, 16, 64, 8
    rng = np.random.default_rng(5)
    ktab = rng.standard_normal((50, n_kv, d))
    vtab = rng.standard_normal((50, n_kv, d))
    bf = lambda x: torch.as_tensor(x, dtype=torch.float32).to(torch.bfloat16)
    kp = torch.zeros(N, n_kv, bs, d, dtype=torch.bfloat16, device=DEV)
    vp = torch.zeros_like(kp)
    kh = torch.zeros(H, n_kv, bs, d, dtype=torch.bfloat16).pin_memory()
    vh = torch.zeros_like(kh).pin_memory()
    bm = pkv.BlockManager(N, bs, host_blocks=H)
    err = err_flag()
    prefixes = [list(rng.integers(0, 50, size=int(rng.integers(bs, 3 * bs)))) for _ in range(3)]
    live = {}
    sid = 0

    def write(toks, positions, slots):
        if not len(slots):
            return
        k = np.stack([_kv_of(toks[p], p, n_kv, d, ktab) for p in positions])
        v = np.stack([_kv_of(toks[p], p, n_kv, d, vtab) for p in positions])
        pkv.kv_append(bf(k).to(DEV), bf(v).to(DEV), torch.as_tensor(np.asarray(slots, np.int64), device=DEV),
                      kp, vp, err=err)

    def apply():
        c = bm.take_copies()
        if len(c):
            pkv.copy_blocks(c, kp, vp, kh, vh)
        return len(c)

    moved = 0
    for step in range(250):
        op = rng.random()
        if op < 0.3 or not live:
            sid += 1
            toks = list(prefixes[int(rng.integers(0, 3))]) + list(rng.integers(0, 50, size=int(rng.integers(1, 20))))
            try:
                table, reused = bm.add_sequence(sid, toks, ranges=[(0, bs, int(rng.integers(20, 90)))])
            except pkv.PkvError:
                moved += apply()
                continue
            moved += apply()
            pos = list(range(reused, len(toks)))
            write(toks, pos, [table[p // bs] * bs + p % bs for p in pos])
            live[sid] = toks
        elif op < 0.8:
            s = list(live)[int(rng.integers(0, len(live)))]
            t = int(rng.integers(0, 50))
            try:
                slot = bm.append_tokens([s], [t])
            except pkv.PkvError:
                moved += apply()
                continue
            moved += apply()
            live[s].append(t)
            write(live[s], [len(live[s]) - 1], slot)
        else:
            s = list(live)[int(rng.integers(0, len(live)))]
            bm.release(s)
            del live[s]
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    c = bm.counts()
    assert moved > 0 and c["onloads"] > 0 and c["offloads"] > 0, c
    seqs = sorted(live)
    mb = max(-(-len(live[s]) // bs) for s in seqs)
    tables, ctx = bm.tables(seqs, mb)
    q = torch.randn(len(seqs), n_h, d, generator=torch.Generator().manual_seed(1)).to(torch.bfloat16)
    out = pkv.paged_decode_attn(q.to(DEV), kp, vp, torch.as_tensor(tables, device=DEV),
                                torch.as_tensor(ctx, device=DEV), 1 / math.sqrt(d), out_dtype=torch.float32,
                                err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    # the oracle on each sequence's own rows, laid out contiguously
    for r, s in enumerate(seqs):
        toks = live[s]
        L = len(toks)
        nb = -(-L // bs)
        k2 = np.zeros((nb, n_kv, bs, d))
        v2 = np.zeros_like(k2)
        for p in range(L):
            k2[p // bs, :, p % bs] = f64(bf(_kv_of(toks[p], p, n_kv, d, ktab)))
            v2[p // bs, :, p % bs] = f64(bf(_kv_of(toks[p], p, n_kv, d, vtab)))
        ref = oracle.paged_decode_attention(f64(q[r:r + 1]), k2, v2, np.arange(nb)[None, :], np.array([L]),
                                            1 / math.sqrt(d), bs)
        check_attention(out[r:r + 1], ref, f"sequence {s}")
