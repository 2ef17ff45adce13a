"""The C-ABI library builds here (cross-compiled for sm_103a), loads, and exports every
entry point include/*.h declares.  No compute calls: this machine has no GPU."""
import os
import re
import subprocess

import pytest

import paged_kv_cache_175_gb300 as pkv
from paged_kv_cache_175_gb300 import _build

INCLUDE = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include")


def _declared():
    names = set()
    for h in sorted(os.listdir(INCLUDE)):
        if h.endswith(".h"):
            text = re.sub(r"/\*.*?\*/", "", open(os.path.join(INCLUDE, h)).read(), flags=re.S)
            names.update(re.findall(r"\b(pkv_[a-z0-9_]+)\s*\(", text))
    return sorted(names)


@pytest.fixture(scope="module")
def built():
    return _build.build_library()


def test_header_declares_the_entry_points():
    names = _declared()
    for n in ("pkv_kv_append", "pkv_paged_decode_attn", "pkv_kv_quant_append_int4",
              "pkv_paged_decode_attn_int4", "pkv_rope_shift_k", "pkv_decode_workspace_bytes",
              "pkv_status_str", "pkv_last_cuda_error", "pkv_paged_decode_attn_window",
              "pkv_paged_decode_attn_int4_window", "pkv_bm_create", "pkv_bm_add_sequence", "pkv_copy_blocks"):
        assert n in names


def test_library_exports_every_declared_symbol(built):
    out = subprocess.run(["nm", "-D", "--defined-only", built], capture_output=True, text=True, check=True).stdout
    exported = set(re.findall(r" T (pkv_\w+)", out))
    missing = [n for n in _declared() if n not in exported]
    assert not missing, missing


def test_library_loads_and_binding_matches_header(built):
    l = pkv.lib()
    for n in _declared():
        assert hasattr(l, n)
        assert n in pkv._SIGS, f"binding lacks {n}"
    assert l.pkv_status_str(0) == b"ok"
    assert l.pkv_status_str(-4) == b"workspace too small"
    assert l.pkv_status_str(7) == b"unknown status"


def test_binding_refuses_cpu_tensors(built):
    import torch
    k = torch.zeros(1, 1, 64, dtype=torch.bfloat16)
    with pytest.raises(pkv.PkvError):
        pkv.kv_append(k, k, torch.zeros(1, dtype=torch.int64), torch.zeros(1, 1, 16, 64, dtype=torch.bfloat16),
                      torch.zeros(1, 1, 16, 64, dtype=torch.bfloat16))


def test_layer_window_is_the_list_repeated_over_the_layers(built):
    # "KV 캐시 시스템 (KV Cache System)", section "어텐션 윈도우 크기": the page's own
    # examples, one window for every layer and [4096, 256] alternating over six layers
    import oracle
    assert pkv.layer_windows([4096], 4) == [4096] * 4
    assert pkv.layer_windows([4096, 256], 6) == [4096, 256, 4096, 256, 4096, 256]
    for lst, n in (([4096, 256, 128], 4), ([7], 1), ([1, 2, 3, 4, 5], 12)):
        assert pkv.layer_windows(lst, n) == oracle.layer_windows(lst, n)
    for bad in ([], [0], [4096, -1]):
        with pytest.raises(ValueError):
            pkv.layer_windows(bad, 3)
    import ctypes
    assert pkv.lib().pkv_layer_window(None, 2, 0) == -1
    w = (ctypes.c_int32 * 2)(8, 16)
    assert pkv.lib().pkv_layer_window(w, 2, -1) == -1
    assert pkv.lib().pkv_layer_window(w, 2, 5) == 16
