"""The HBM ceiling probes: the copy probe copies every byte, the read probe writes nothing,
and bad arguments are refused before anything is launched."""
import ctypes

import pytest
import torch

import paged_kv_cache_175_gb300 as pkv

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("nbytes", [16, 4096 + 48, (1 << 24) + 16 * 7])
def test_copy_probe_copies_every_byte(nbytes):
    g = torch.Generator(device="cuda").manual_seed(nbytes)
    src = torch.randint(0, 256, (nbytes,), dtype=torch.uint8, device="cuda", generator=g)
    dst = torch.zeros_like(src)
    pkv.probe_copy(src, dst)
    torch.cuda.synchronize()
    assert torch.equal(src, dst)


def test_read_probe_leaves_its_buffer_and_sink_alone():
    buf = torch.arange(1 << 22, dtype=torch.int32, device="cuda")
    before = buf.clone()
    sink = torch.full((1,), 7, dtype=torch.int32, device="cuda")
    pkv.probe_read(buf, sink=sink)
    pkv.probe_read(buf)
    torch.cuda.synchronize()
    assert torch.equal(buf, before) and int(sink.item()) == 7


def test_probe_arguments_are_checked():
    l = pkv.lib()
    buf = torch.zeros(64, dtype=torch.uint8, device="cuda")
    p = ctypes.c_void_p(buf.data_ptr())
    assert l.pkv_probe_read(p, 24, None, None) == -1                            # not a multiple of 16
    assert l.pkv_probe_read(ctypes.c_void_p(buf.data_ptr() + 4), 16, None, None) == -1   # misaligned
    assert l.pkv_probe_read(None, 16, None, None) == -1
    assert l.pkv_probe_copy(p, ctypes.c_void_p(buf.data_ptr() + 16), 32, None) == -1     # overlapping
    assert l.pkv_probe_copy(p, ctypes.c_void_p(buf.data_ptr() + 32), 32, None) == 0
    torch.cuda.synchronize()
