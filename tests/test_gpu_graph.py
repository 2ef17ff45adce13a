"""A decode step (append + attention) captured in a CUDA graph and replayed gives the same
bits as the same calls launched eagerly (bf16 and INT4 caches), and repeated calls give the
same bits."""
import numpy as np
import pytest
import torch

import paged_kv_cache_175_gb300 as pkv
import workloads
from gpu_common import DEV, err_flag

pytestmark = pytest.mark.gpu


def test_bf16_step_graph_equals_eager():
    w = workloads.make("llama3_8b_b16", 0)
    kp, vp = workloads.pools_bf16(w, 0, DEV)
    kp2, vp2 = kp.clone(), vp.clone()
    q = workloads.queries(w, 0, DEV)
    kn, vn = workloads.new_tokens(w, 0, DEV)
    slots = torch.as_tensor(workloads.decode_slots(w), device=DEV)
    bt = torch.as_tensor(w.block_tables, device=DEV)
    ctx = torch.as_tensor(w.context_lens, device=DEV)
    ws = torch.empty(pkv.decode_workspace_bytes(w.batch, w.n_h, w.n_kv, w.head_dim, w.block_size),
                     dtype=torch.uint8, device=DEV)
    err = err_flag()
    out_e, out_g = torch.empty_like(q), torch.empty_like(q)

    def step(k_pool, v_pool, out):
        pkv.kv_append(kn, vn, slots, k_pool, v_pool, err=err)
        pkv.paged_decode_attn(q, k_pool, v_pool, bt, ctx, w.scale, out=out, workspace=ws, err=err)

    step(kp, vp, out_e)                                    # eager (also sets up the kernels)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step(kp2, vp2, out_g)
    g.replay()
    g.replay()                                            # replays are idempotent here
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert torch.equal(out_e, out_g) and torch.equal(kp, kp2) and torch.equal(vp, vp2)


def test_int4_step_graph_equals_eager():
    w = workloads.make("int4_long_b8", 0)
    bs = w.block_size
    caches = [pkv.alloc_int4_cache(w.num_blocks, w.n_kv, bs, w.head_dim, w.batch, DEV) for _ in range(2)]
    ks, vs, sl, tl, newk, newv = [], [], [], [], [], []
    for s in range(w.batch):
        k, v = workloads.history_kv(w, s, 0, DEV)
        slots = workloads.history_slots(w, s)
        ks.append(k[:-1]); vs.append(v[:-1]); sl.append(slots[:-1]); tl.append(np.full(len(slots) - 1, s, np.int32))
        newk.append(k[-1]); newv.append(v[-1])
    for c in caches:
        pkv.kv_quant_append_int4(torch.cat(ks), torch.cat(vs), torch.as_tensor(np.concatenate(sl), device=DEV),
                                 torch.as_tensor(np.concatenate(tl), device=DEV), c)
    kn, vn = torch.stack(newk).contiguous(), torch.stack(newv).contiguous()
    slots = torch.as_tensor(workloads.decode_slots(w), device=DEV)
    tails = torch.arange(w.batch, dtype=torch.int32, device=DEV)
    q = workloads.queries(w, 0, DEV)
    bt = torch.as_tensor(w.block_tables, device=DEV)
    ctx = torch.as_tensor(w.context_lens, device=DEV)
    ws = torch.empty(pkv.decode_workspace_bytes(w.batch, w.n_h, w.n_kv, w.head_dim, bs, int4=True),
                     dtype=torch.uint8, device=DEV)
    err = err_flag()
    out_e, out_g = torch.empty_like(q), torch.empty_like(q)

    def step(cache, out):
        pkv.kv_quant_append_int4(kn, vn, slots, tails, cache, err=err)
        pkv.paged_decode_attn_int4(q, cache, bt, ctx, w.scale, out=out, workspace=ws, err=err)

    step(caches[0], out_e)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step(caches[1], out_g)
    g.replay()
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert torch.equal(out_e, out_g)
    for a, b in zip((caches[0].k_codes, caches[0].v_codes, caches[0].k_meta, caches[0].v_meta, caches[0].k_tail),
                    (caches[1].k_codes, caches[1].v_codes, caches[1].k_meta, caches[1].v_meta, caches[1].k_tail)):
        assert torch.equal(a, b)


@pytest.mark.parametrize("name", ["mqa_bs16", "llama3_8b_b16"])
def test_repeated_calls_are_bitwise_identical(name):
    """The partition, the ring and the merge order are fixed, so repeated calls give the same
    bits (a race on a reused ring slot would show up here as a difference)."""
    w = workloads.make(name, 0)
    kp, vp = workloads.pools_bf16(w, 0, DEV)
    q = workloads.queries(w, 0, DEV)
    bt = torch.as_tensor(w.block_tables, device=DEV)
    ctx = torch.as_tensor(w.context_lens, device=DEV)
    err = err_flag()
    ref = pkv.paged_decode_attn(q, kp, vp, bt, ctx, w.scale, out_dtype=torch.float32, err=err)
    outs = [pkv.paged_decode_attn(q, kp, vp, bt, ctx, w.scale, out_dtype=torch.float32, err=err) for _ in range(20)]
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert all(torch.equal(o, ref) for o in outs)


def test_repeated_int4_calls_are_bitwise_identical():
    w = workloads.make("int4_long_b8", 0)
    bs = w.block_size
    cache = pkv.alloc_int4_cache(w.num_blocks, w.n_kv, bs, w.head_dim, w.batch, DEV)
    ks, vs, sl, tl = [], [], [], []
    for s in range(w.batch):
        k, v = workloads.history_kv(w, s, 0, DEV)
        slots = workloads.history_slots(w, s)
        ks.append(k); vs.append(v); sl.append(slots); tl.append(np.full(len(slots), s, np.int32))
    pkv.kv_quant_append_int4(torch.cat(ks), torch.cat(vs), torch.as_tensor(np.concatenate(sl), device=DEV),
                             torch.as_tensor(np.concatenate(tl), device=DEV), cache)
    q = workloads.queries(w, 0, DEV)
    bt = torch.as_tensor(w.block_tables, device=DEV)
    ctx = torch.as_tensor(w.context_lens, device=DEV)
    err = err_flag()
    ref = pkv.paged_decode_attn_int4(q, cache, bt, ctx, w.scale, out_dtype=torch.float32, err=err)
    outs = [pkv.paged_decode_attn_int4(q, cache, bt, ctx, w.scale, out_dtype=torch.float32, err=err)
            for _ in range(20)]
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert all(torch.equal(o, ref) for o in outs)
