"""The allocation-free decode entry point, called through the C ABI.

pkv_paged_decode_attn_noalloc serves callers that cannot allocate device memory while
they decode; its scratch is a fixed array inside the library.  Two calls in a row (with
different shapes, so the second one runs over whatever the first left in the shared
array) must give the same output as pkv_paged_decode_attn with a caller workspace,
within the tolerance the other attention tests use.  This file is collected last so a
run that stops at the first failure has already run every other test.
"""
import ctypes
import math

import numpy as np
import pytest
import torch

import paged_kv_cache_175_gb300 as pkv
import workloads
from gpu_common import BAR_F32_MAXABS, BAR_F32_RELL2, DEV, f64, rel_l2
from paged_kv_cache_175_gb300._build import build_library

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def library():
    build_library()
    return pkv.lib()


def _case(name_or_shape, seed):
    if isinstance(name_or_shape, str):
        w = workloads.make(name_or_shape, seed)
        kp, vp = workloads.pools_bf16(w, seed, DEV)
        q = workloads.queries(w, seed, DEV)
        return q, kp, vp, w.block_tables, w.context_lens, w.scale
    D, BS, n_h, n_kv, ctx = name_or_shape
    rng = np.random.default_rng(seed)
    nbs = [-(-c // BS) for c in ctx]
    num_blocks = sum(nbs) + 3
    perm = rng.permutation(num_blocks).astype(np.int32)
    bt = np.full((len(ctx), max(nbs)), -1, dtype=np.int32)
    cur = 0
    for s, n in enumerate(nbs):
        bt[s, :n] = perm[cur:cur + n]
        cur += n
    g = torch.Generator(device=DEV).manual_seed(seed)
    kp = torch.randn(num_blocks, n_kv, BS, D, generator=g, device=DEV).to(torch.bfloat16)
    vp = torch.randn(num_blocks, n_kv, BS, D, generator=g, device=DEV).to(torch.bfloat16)
    q = torch.randn(len(ctx), n_h, D, generator=g, device=DEV).to(torch.bfloat16)
    return q, kp, vp, bt, np.asarray(ctx, dtype=np.int32), 1 / math.sqrt(D)


def _noalloc_c_call(lib, q, kp, vp, bt, ctx, scale, out, err):
    num_blocks, n_kv, bs, d = kp.shape
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    return lib.pkv_paged_decode_attn_noalloc(
        p(q), p(kp), p(vp), p(bt), bt.shape[1], p(ctx), ctypes.c_float(scale), q.shape[0], q.shape[1], n_kv, d, bs,
        num_blocks, p(out), pkv.PKV_OUT_F32 if out.dtype == torch.float32 else pkv.PKV_OUT_BF16, p(err),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_two_calls_in_a_row_match_the_workspace_entry_point(library, out_dtype):
    cases = ["llama3_8b", (64, 32, 8, 2, [1, 40, 300, 31])]
    for i, c in enumerate(cases):
        q, kp, vp, bt, ctx, scale = _case(c, seed=i)
        btd, ctxd = torch.as_tensor(bt, device=DEV), torch.as_tensor(ctx, device=DEV)
        err = torch.zeros(1, dtype=torch.int32, device=DEV)
        out = torch.full(q.shape, float("nan"), dtype=out_dtype, device=DEV)
        st = _noalloc_c_call(library, q, kp, vp, btd, ctxd, scale, out, err)
        assert st == 0, library.pkv_status_str(st)
        ref = pkv.paged_decode_attn(q, kp, vp, btd, ctxd, scale, out_dtype=out_dtype, err=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        a, b = f64(out), f64(ref)
        assert np.isfinite(a).all()
        assert np.abs(a - b).max() <= BAR_F32_MAXABS and rel_l2(a, b) <= BAR_F32_RELL2, (c, out_dtype)


def test_shape_beyond_the_static_scratch_is_rejected(library):
    # 4096 sequences x 64 query heads need far more than the fixed scratch: the call
    # returns PKV_ERANGE before touching any pointer or launching anything
    need = library.pkv_decode_workspace_bytes(4096, 64, 1, 128, 16, 0)
    assert need > pkv.STATIC_SCRATCH_BYTES
    st = library.pkv_paged_decode_attn_noalloc(None, None, None, None, 1, None, ctypes.c_float(0.1), 4096, 64, 1,
                                               128, 16, 1, None, 0, None, None)
    assert st == -2 and library.pkv_status_str(st) == b"size out of range"


def test_python_wrapper_against_the_oracle(library):
    # the tiny workload through pkv.paged_decode_attn_noalloc, checked against the fp64
    # oracle with the bars of the other attention tests (bf16 and fp32 output)
    import oracle
    from gpu_common import check_attention
    w = workloads.make("tiny", 0)
    kp, vp = workloads.pools_bf16(w, 0, DEV)
    q = workloads.queries(w, 0, DEV)
    ref = oracle.paged_decode_attention(f64(q), f64(kp), f64(vp), w.block_tables, w.context_lens, w.scale,
                                        w.block_size)
    for od in (torch.bfloat16, torch.float32):
        err = torch.zeros(1, dtype=torch.int32, device=DEV)
        out = pkv.paged_decode_attn_noalloc(q, kp, vp, torch.as_tensor(w.block_tables, device=DEV),
                                            torch.as_tensor(w.context_lens, device=DEV), w.scale, out_dtype=od,
                                            err=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        check_attention(out, ref, f"noalloc tiny {od}")
    with pytest.raises(AssertionError):                  # int64 tables are refused, not misread
        pkv.paged_decode_attn_noalloc(q, kp, vp, torch.as_tensor(w.block_tables, device=DEV).long(),
                                      torch.as_tensor(w.context_lens, device=DEV), w.scale)
