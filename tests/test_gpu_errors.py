"""Argument checks of the C ABI (bad shapes and sizes return an error, nothing is launched)
and the device-side failure detection of the bounded waits."""
import pytest
import torch

import paged_kv_cache_175_gb300 as pkv
from gpu_common import DEV

pytestmark = pytest.mark.gpu


def _call(**over):
    a = dict(q=torch.zeros(2, 8, 128, dtype=torch.bfloat16, device=DEV),
             k=torch.zeros(4, 2, 16, 128, dtype=torch.bfloat16, device=DEV),
             bt=torch.zeros(2, 2, dtype=torch.int32, device=DEV),
             ctx=torch.tensor([3, 4], dtype=torch.int32, device=DEV))
    a.update(over)
    return pkv.paged_decode_attn(a["q"], a["k"], a["k"], a["bt"], a["ctx"], 0.1,
                                 workspace=a.get("ws"))


def test_valid_call_runs():
    out = _call()
    torch.cuda.synchronize()
    assert out.shape == (2, 8, 128)


@pytest.mark.parametrize("case", ["head_dim", "block_size", "group", "too_many_groups"])
def test_bad_shapes_are_rejected(case):
    if case == "head_dim":
        kw = dict(q=torch.zeros(2, 8, 96, dtype=torch.bfloat16, device=DEV),
                  k=torch.zeros(4, 2, 16, 96, dtype=torch.bfloat16, device=DEV))
    elif case == "block_size":
        kw = dict(k=torch.zeros(4, 2, 8, 128, dtype=torch.bfloat16, device=DEV))
    elif case == "group":
        kw = dict(k=torch.zeros(4, 3, 16, 128, dtype=torch.bfloat16, device=DEV))
    else:
        kw = dict(q=torch.zeros(2, 128, 128, dtype=torch.bfloat16, device=DEV),
                  k=torch.zeros(4, 1, 16, 128, dtype=torch.bfloat16, device=DEV))
    with pytest.raises(pkv.PkvError):
        _call(**kw)


def test_small_workspace_is_rejected():
    with pytest.raises(pkv.PkvError, match="workspace too small"):
        _call(ws=torch.empty(256, dtype=torch.uint8, device=DEV))


def test_misaligned_pointer_is_rejected():
    buf = torch.zeros(2 * 8 * 128 + 1, dtype=torch.bfloat16, device=DEV)
    q = buf[1:].view(2, 8, 128)                                  # 2-byte offset
    with pytest.raises(pkv.PkvError, match="invalid argument"):
        _call(q=q)


def test_empty_batch_is_a_no_op():
    out = _call(q=torch.zeros(0, 8, 128, dtype=torch.bfloat16, device=DEV),
                bt=torch.zeros(0, 2, dtype=torch.int32, device=DEV),
                ctx=torch.zeros(0, dtype=torch.int32, device=DEV))
    assert out.shape == (0, 8, 128)


def test_bounded_wait_runs_out_and_the_context_stays_usable():
    """A wait on a barrier nobody arrives at gives up after its limit and reports
    DEV_TIMEOUT through the flag; a wait whose arrival came first reports nothing; the next
    attention call on the same context is still correct."""
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    pkv.selftest_wait(True, 1000, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    pkv.selftest_wait(False, 2000, err)
    torch.cuda.synchronize()
    assert int(err.item()) == pkv.DEV_TIMEOUT
    with pytest.raises(pkv.PkvError):
        pkv.selftest_wait(False, 0, err)
    import numpy as np
    import oracle
    import workloads
    from gpu_common import check_attention, f64, run_attention
    w = workloads.make("tiny", 0)
    kp, vp = workloads.pools_bf16(w, 0)
    q = workloads.queries(w, 0)
    ref = oracle.paged_decode_attention(f64(q), f64(kp), f64(vp), w.block_tables, w.context_lens, w.scale,
                                        w.block_size)
    out = run_attention(q.to(DEV), kp.to(DEV), vp.to(DEV), w.block_tables, w.context_lens, w.scale, torch.float32)
    check_attention(out, ref, "after a timed-out wait")
