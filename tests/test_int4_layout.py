"""Host-side checks of the INT4 cache record layout (no GPU): the record size the library
reports, and the four field views of the Python cache object over one record."""
import numpy as np
import pytest
import torch

import paged_kv_cache_175_gb300 as pkv


@pytest.mark.parametrize("bs", [16, 32, 64])
@pytest.mark.parametrize("d", [64, 128])
def test_record_bytes(bs, d):
    r = pkv.int4_record_bytes(bs, d)
    assert r == bs * d + 4 * d + 4 * bs          # codes of K and V, K scale+min rows, V (scale, min) per token
    assert r % 16 == 0                           # one bulk copy per record needs 16-byte multiples


@pytest.mark.parametrize("bs,d", [(8, 128), (16, 96), (128, 64), (0, 128)])
def test_record_bytes_rejects_other_shapes(bs, d):
    assert pkv.int4_record_bytes(bs, d) == 0
    with pytest.raises(ValueError):
        pkv.alloc_int4_cache(4, 2, bs, d, 1, "cpu")


@pytest.mark.parametrize("bs,d", [(16, 128), (64, 64)])
def test_field_views_cover_each_record_once(bs, d):
    nb, n_kv = 3, 2
    c = pkv.alloc_int4_cache(nb, n_kv, bs, d, 1, "cpu")
    r = pkv.int4_record_bytes(bs, d)
    assert tuple(c.records.shape) == (nb, n_kv, r) and c.shape == (nb, n_kv, bs, d)
    assert c.k_codes.shape == (nb, n_kv, bs, d // 2) and c.v_codes.shape == (nb, n_kv, bs, d // 2)
    assert c.k_meta.shape == (nb, n_kv, 2, d) and c.k_meta.dtype == torch.float16
    assert c.v_meta.shape == (nb, n_kv, bs, 2) and c.v_meta.dtype == torch.float16
    # distinct bytes everywhere: each field must read its own slice of its own record
    rng = np.random.default_rng(0)
    c.records.copy_(torch.as_tensor(rng.integers(0, 256, size=c.records.shape, dtype=np.uint8)))
    raw = c.records.numpy()
    for b in range(nb):
        for g in range(n_kv):
            rec = raw[b, g]
            assert c.k_codes[b, g].numpy().tobytes() == rec[:bs * d // 2].tobytes()
            assert c.v_codes[b, g].numpy().tobytes() == rec[bs * d // 2:bs * d].tobytes()
            assert c.k_meta[b, g].numpy().tobytes() == rec[bs * d:bs * d + 4 * d].tobytes()
            assert c.v_meta[b, g].numpy().tobytes() == rec[bs * d + 4 * d:].tobytes()
    # the views alias the records (writes through a view land in the record)
    c.v_meta[1, 1, 0, 1] = 2.5
    assert np.frombuffer(raw[1, 1, bs * d + 4 * d + 2:bs * d + 4 * d + 4].tobytes(), np.float16)[0] == 2.5
