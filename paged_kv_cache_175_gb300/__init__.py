"""Python binding of libpkv.so — paged KV-cache decode attention for GB300 (sm_103a).

Argument marshalling only: every step of the computation runs in the CUDA library
(see include/pkv.h for the contract of each call).  torch supplies device memory
and streams.  There is no CPU fallback: the calls raise if the library is not
built or a tensor is not on a CUDA device.

Functions (same names as the C entry points without the ``pkv_`` prefix):
``kv_append``, ``paged_decode_attn``, ``paged_decode_attn_window``,
``paged_decode_attn_noalloc``, ``kv_quant_append_int4``, ``paged_decode_attn_int4``,
``paged_decode_attn_int4_window``, ``rope_shift_k``, ``copy_blocks``, ``kv_deviation``,
``select_top``, ``kv_fuse``, ``recompute_ratio``, ``select_count``, ``probe_read``,
``probe_copy``, ``layer_window`` (as ``layer_windows``), plus
``decode_workspace_bytes``, ``alloc_int4_cache`` and ``BlockManager`` (the ``pkv_bm_*`` calls of include/pkv_bm.h).
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import torch

from ._build import LIB as LIB_PATH, build_library

PKV_OUT_BF16 = 0
PKV_OUT_F32 = 1
DEV_BAD_BLOCK, DEV_BAD_SLOT, DEV_BAD_CTX, DEV_TIMEOUT = 1, 2, 4, 8

_lib = None

_P = ctypes.c_void_p
_I = ctypes.c_int
_SIGS = {
    "pkv_status_str": (ctypes.c_char_p, [_I]),
    "pkv_last_cuda_error": (_I, []),
    "pkv_kv_append": (_I, [_P, _P, _P, _I, _P, _P, _I, _I, _I, _I, _P, _P]),
    "pkv_decode_workspace_bytes": (ctypes.c_size_t, [_I, _I, _I, _I, _I, _I]),
    "pkv_paged_decode_attn": (_I, [_P, _P, _P, _P, _I, _P, ctypes.c_float, _I, _I, _I, _I, _I, _I,
                                   _P, _I, _P, ctypes.c_size_t, _P, _P]),
    "pkv_kv_quant_append_int4": (_I, [_P, _P, _P, _P, _I, _P, _P, _I, _I, _I, _I, _I, _P, _P]),
    "pkv_int4_record_bytes": (ctypes.c_size_t, [_I, _I]),
    "pkv_paged_decode_attn_int4": (_I, [_P, _P, _P, _P, _I, _P, ctypes.c_float, _I, _I, _I, _I, _I, _I,
                                        _P, _I, _P, ctypes.c_size_t, _P, _P]),
    "pkv_rope_shift_k": (_I, [_P, _P, _P, _I, _I, _I, _I, _I, ctypes.c_double, _P, _P]),
    "pkv_paged_decode_attn_noalloc": (_I, [_P, _P, _P, _P, _I, _P, ctypes.c_float, _I, _I, _I, _I, _I, _I,
                                           _P, _I, _P, _P]),
    "pkv_paged_decode_attn_window": (_I, [_P, _P, _P, _P, _I, _P, ctypes.c_float, _I, _I, _I, _I, _I, _I, _I,
                                          _P, _I, _P, ctypes.c_size_t, _P, _P]),
    "pkv_paged_decode_attn_int4_window": (_I, [_P, _P, _P, _P, _I, _P, ctypes.c_float, _I, _I, _I, _I, _I, _I,
                                               _I, _P, _I, _P, ctypes.c_size_t, _P, _P]),
    # block manager (host) and its copy executor
    "pkv_bm_create": (_P, [_I, _I, _I, _I, _I]),
    "pkv_bm_destroy": (None, [_P]),
    "pkv_bm_add_sequence": (_I, [_P, ctypes.c_int64, _P, _I, _P, _I, _P, _I]),
    "pkv_bm_append_tokens": (_I, [_P, _P, _P, _I, _P, _P]),
    "pkv_bm_release": (_I, [_P, ctypes.c_int64]),
    "pkv_bm_slide_window": (_I, [_P, ctypes.c_int64, _I]),
    "pkv_bm_tables": (_I, [_P, _P, _I, _P, _I, _P]),
    "pkv_bm_take_copies": (_I, [_P, _P, _I]),
    "pkv_bm_pending_copies": (_I, [_P]),
    "pkv_bm_counts": (None, [_P, _P]),
    "pkv_copy_blocks": (_I, [_P, _I, _P, _P, _I, _P, _P, _I, ctypes.c_size_t, _P]),
    # CacheBlend's model-free steps
    "pkv_kv_deviation": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _P, _P]),
    "pkv_select_top": (_I, [_P, _P, _P, _I, _P, _P]),
    "pkv_kv_fuse": (_I, [_P, _P, _P, _I, _P, _I, _P, _P, _I, _I, _I, _I, _P, _P]),
    "pkv_recompute_ratio": (ctypes.c_double, [ctypes.c_double, ctypes.c_double]),
    "pkv_select_count": (_I, [ctypes.c_double, _I]),
    "pkv_selftest_wait": (_I, [_I, _I, _P, _P]),
    "pkv_layer_window": (_I, [_P, _I, _I]),
    "pkv_probe_read": (_I, [_P, ctypes.c_size_t, _P, _P]),
    "pkv_probe_copy": (_I, [_P, _P, ctypes.c_size_t, _P]),
}
STATIC_SCRATCH_BYTES = 16 * 1024 * 1024


class PkvError(RuntimeError):
    pass


def lib(build_if_missing: bool = False) -> ctypes.CDLL:
    """Load libpkv.so (fails loudly if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            if not build_if_missing:
                raise PkvError(f"{LIB_PATH} is missing: build it with paged_kv_cache_175_gb300._build.build_library()")
            build_library()
        l = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            f = getattr(l, name)
            f.restype = res
            f.argtypes = args
        _lib = l
    return _lib


def _check(name: str, status: int):
    if status != 0:
        msg = lib().pkv_status_str(status).decode()
        extra = f" (cuda error {lib().pkv_last_cuda_error()})" if status == -3 else ""
        raise PkvError(f"{name}: {msg}{extra}")


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _cuda(*ts):
    for t in ts:
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise PkvError("tensors must be contiguous CUDA tensors")


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def kv_append(k, v, slot_mapping, k_pool, v_pool, err=None, stream=None):
    """Write k, v [n_tok][n_kv][d] (bf16) into the pools at slot_mapping (int64)."""
    _cuda(k, v, slot_mapping, k_pool, v_pool, err)
    assert k.dtype == v.dtype == k_pool.dtype == v_pool.dtype == torch.bfloat16
    assert slot_mapping.dtype == torch.int64
    num_blocks, n_kv, bs, d = k_pool.shape
    _check("kv_append", lib().pkv_kv_append(_ptr(k), _ptr(v), _ptr(slot_mapping), k.shape[0], _ptr(k_pool),
                                            _ptr(v_pool), num_blocks, bs, n_kv, d, _ptr(err), _stream(stream)))


def decode_workspace_bytes(batch, n_h, n_kv, head_dim, block_size, int4=False) -> int:
    n = lib().pkv_decode_workspace_bytes(batch, n_h, n_kv, head_dim, block_size, 1 if int4 else 0)
    if n == 0 and batch > 0:
        raise PkvError("decode_workspace_bytes: invalid shape or no device")
    return n


def _workspace(nbytes, device):
    return torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)


def _out(q, out, out_dtype):
    if out is None:
        out = torch.empty(q.shape, dtype=out_dtype, device=q.device)
    assert out.shape == q.shape and out.dtype in (torch.bfloat16, torch.float32)
    return out, (PKV_OUT_F32 if out.dtype == torch.float32 else PKV_OUT_BF16)


def paged_decode_attn(q, k_pool, v_pool, block_tables, context_lens, scale, out=None, out_dtype=torch.bfloat16,
                      workspace=None, err=None, stream=None):
    """Decode attention over a paged bf16 cache; returns out [B][n_h][d]."""
    return _decode_bf16(q, k_pool, v_pool, block_tables, context_lens, scale, 0, out, out_dtype, workspace, err,
                        stream)


def paged_decode_attn_window(q, k_pool, v_pool, block_tables, context_lens, scale, window, out=None,
                             out_dtype=torch.bfloat16, workspace=None, err=None, stream=None):
    """Decode attention over the last `window` tokens of each context (0: all of it)."""
    return _decode_bf16(q, k_pool, v_pool, block_tables, context_lens, scale, int(window), out, out_dtype,
                        workspace, err, stream)


def layer_windows(max_attention_window, n_layers):
    """Attention window of each of n_layers layers from a max_attention_window list
    (pkv_layer_window: the list repeated over the layers)."""
    import numpy as np
    w = np.ascontiguousarray(max_attention_window, dtype=np.int32).reshape(-1)
    out = [lib().pkv_layer_window(w.ctypes.data, len(w), i) for i in range(max(int(n_layers), 1))]
    if any(x < 0 for x in out):
        raise ValueError("max_attention_window must be a non-empty list of positive token counts")
    return out[:int(n_layers)]


def _decode_bf16(q, k_pool, v_pool, block_tables, context_lens, scale, window, out, out_dtype, workspace, err,
                 stream):
    _cuda(q, k_pool, v_pool, block_tables, context_lens, out, workspace, err)
    assert q.dtype == k_pool.dtype == v_pool.dtype == torch.bfloat16
    assert block_tables.dtype == context_lens.dtype == torch.int32
    B, n_h, d = q.shape
    num_blocks, n_kv, bs, d2 = k_pool.shape
    assert d2 == d and v_pool.shape == k_pool.shape
    out, od = _out(q, out, out_dtype)
    need = decode_workspace_bytes(B, n_h, n_kv, d, bs)
    if workspace is None:
        workspace = _workspace(need, q.device)
    if window == 0:
        _check("paged_decode_attn", lib().pkv_paged_decode_attn(
            _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(block_tables), block_tables.shape[1], _ptr(context_lens),
            float(scale), B, n_h, n_kv, d, bs, num_blocks, _ptr(out), od, _ptr(workspace), workspace.numel(),
            _ptr(err), _stream(stream)))
    else:
        _check("paged_decode_attn_window", lib().pkv_paged_decode_attn_window(
            _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(block_tables), block_tables.shape[1], _ptr(context_lens),
            float(scale), window, B, n_h, n_kv, d, bs, num_blocks, _ptr(out), od, _ptr(workspace),
            workspace.numel(), _ptr(err), _stream(stream)))
    return out


def paged_decode_attn_noalloc(q, k_pool, v_pool, block_tables, context_lens, scale, out=None,
                              out_dtype=torch.bfloat16, err=None, stream=None):
    """paged_decode_attn with the library's fixed internal scratch instead of a workspace
    (for callers that cannot allocate device memory; concurrent calls must not overlap)."""
    _cuda(q, k_pool, v_pool, block_tables, context_lens, out, err)
    assert q.dtype == k_pool.dtype == v_pool.dtype == torch.bfloat16
    assert block_tables.dtype == context_lens.dtype == torch.int32
    B, n_h, d = q.shape
    num_blocks, n_kv, bs, d2 = k_pool.shape
    assert d2 == d and v_pool.shape == k_pool.shape
    assert block_tables.dim() == 2 and block_tables.shape[0] == B and context_lens.shape == (B,)
    out, od = _out(q, out, out_dtype)
    _check("paged_decode_attn_noalloc", lib().pkv_paged_decode_attn_noalloc(
        _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(block_tables), block_tables.shape[1], _ptr(context_lens),
        float(scale), B, n_h, n_kv, d, bs, num_blocks, _ptr(out), od, _ptr(err), _stream(stream)))
    return out


def int4_record_bytes(block_size, head_dim) -> int:
    """Bytes of one (block, kv head) record of the INT4 cache (0 for an unsupported shape)."""
    return int(lib().pkv_int4_record_bytes(int(block_size), int(head_dim)))


@dataclass
class Int4CacheTensors:
    """INT4 paged cache: one record per (block, kv head) -- K codes, V codes, K scale and
    min rows, V (scale, min) per token -- plus the bf16 K rows of unfinished blocks.  The
    four fields of the records are exposed as views."""
    records: torch.Tensor     # uint8 [num_blocks][n_kv][int4_record_bytes(bs, d)]
    k_tail: torch.Tensor      # bf16  [tail_rows][n_kv][bs][d]

    @property
    def shape(self):
        _, n_kv, bs, d = self.k_tail.shape
        return self.records.shape[0], n_kv, bs, d

    def _field(self, start, size):
        return self.records[:, :, start:start + size]

    @property
    def k_codes(self):         # uint8 [num_blocks][n_kv][bs][d/2]
        nb, n_kv, bs, d = self.shape
        return self._field(0, bs * d // 2).view(nb, n_kv, bs, d // 2)

    @property
    def v_codes(self):         # uint8 [num_blocks][n_kv][bs][d/2]
        nb, n_kv, bs, d = self.shape
        return self._field(bs * d // 2, bs * d // 2).view(nb, n_kv, bs, d // 2)

    @property
    def k_meta(self):          # fp16 [num_blocks][n_kv][2][d]: scale row, min row
        nb, n_kv, bs, d = self.shape
        return self._field(bs * d, 4 * d).view(torch.float16).view(nb, n_kv, 2, d)

    @property
    def v_meta(self):          # fp16 [num_blocks][n_kv][bs][2]: (scale, min) per token
        nb, n_kv, bs, d = self.shape
        return self._field(bs * d + 4 * d, 4 * bs).view(torch.float16).view(nb, n_kv, bs, 2)


def alloc_int4_cache(num_blocks, n_kv, block_size, head_dim, tail_rows, device="cuda") -> Int4CacheTensors:
    rec = int4_record_bytes(block_size, head_dim)
    if rec == 0:
        raise ValueError(f"INT4 cache: unsupported block_size {block_size} / head_dim {head_dim}")
    return Int4CacheTensors(torch.zeros(num_blocks, n_kv, rec, dtype=torch.uint8, device=device),
                            torch.zeros(tail_rows, n_kv, block_size, head_dim, dtype=torch.bfloat16, device=device))


def kv_quant_append_int4(k, v, slot_mapping, tail_seq, cache: Int4CacheTensors, err=None, stream=None):
    """Quantize-on-append of k, v [n_tok][n_kv][d] into the INT4 cache."""
    _cuda(k, v, slot_mapping, tail_seq, cache.records, cache.k_tail, err)
    assert k.dtype == v.dtype == torch.bfloat16 and slot_mapping.dtype == torch.int64
    assert tail_seq.dtype == torch.int32
    nb, n_kv, bs, d = cache.shape
    _check("kv_quant_append_int4", lib().pkv_kv_quant_append_int4(
        _ptr(k), _ptr(v), _ptr(slot_mapping), _ptr(tail_seq), k.shape[0], _ptr(cache.records), _ptr(cache.k_tail),
        cache.k_tail.shape[0], nb, bs, n_kv, d, _ptr(err), _stream(stream)))


def paged_decode_attn_int4(q, cache: Int4CacheTensors, block_tables, context_lens, scale, out=None,
                           out_dtype=torch.bfloat16, workspace=None, err=None, stream=None):
    """Decode attention over the INT4 cache; the batch index is the tail row."""
    return _decode_int4(q, cache, block_tables, context_lens, scale, 0, out, out_dtype, workspace, err, stream)


def paged_decode_attn_int4_window(q, cache: Int4CacheTensors, block_tables, context_lens, scale, window, out=None,
                                  out_dtype=torch.bfloat16, workspace=None, err=None, stream=None):
    """INT4 decode attention over the last `window` tokens of each context (0: all of it)."""
    return _decode_int4(q, cache, block_tables, context_lens, scale, int(window), out, out_dtype, workspace, err,
                        stream)


def _decode_int4(q, cache, block_tables, context_lens, scale, window, out, out_dtype, workspace, err, stream):
    _cuda(q, block_tables, context_lens, out, workspace, err)
    assert q.dtype == torch.bfloat16
    B, n_h, d = q.shape
    nb, n_kv, bs, d2 = cache.shape
    assert d2 == d and cache.k_tail.shape[0] >= B
    out, od = _out(q, out, out_dtype)
    need = decode_workspace_bytes(B, n_h, n_kv, d, bs, int4=True)
    if workspace is None:
        workspace = _workspace(need, q.device)
    if window == 0:
        _check("paged_decode_attn_int4", lib().pkv_paged_decode_attn_int4(
            _ptr(q), _ptr(cache.records), _ptr(cache.k_tail), _ptr(block_tables), block_tables.shape[1],
            _ptr(context_lens), float(scale), B, n_h, n_kv, d, bs, nb, _ptr(out), od, _ptr(workspace), workspace.numel(), _ptr(err), _stream(stream)))
    else:
        _check("paged_decode_attn_int4_window", lib().pkv_paged_decode_attn_int4_window(
            _ptr(q), _ptr(cache.records), _ptr(cache.k_tail), _ptr(block_tables), block_tables.shape[1],
            _ptr(context_lens), float(scale), window, B, n_h, n_kv, d, bs, nb, _ptr(out), od, _ptr(workspace), workspace.numel(), _ptr(err),
            _stream(stream)))
    return out


def rope_shift_k(k_pool, block_ids, deltas, rope_base=10000.0, err=None, stream=None):
    """Rotate every key of block block_ids[i] by position deltas[i] in place."""
    _cuda(k_pool, block_ids, deltas, err)
    assert k_pool.dtype == torch.bfloat16 and block_ids.dtype == deltas.dtype == torch.int32
    num_blocks, n_kv, bs, d = k_pool.shape
    _check("rope_shift_k", lib().pkv_rope_shift_k(_ptr(k_pool), _ptr(block_ids), _ptr(deltas), block_ids.numel(),
                                                  num_blocks, n_kv, bs, d, float(rope_base), _ptr(err),
                                                  _stream(stream)))


# ---------------------------------------------------------------------------------------------
# Block manager (host, include/pkv_bm.h) and the GPU copies it records.
COPY_OFFLOAD, COPY_ONLOAD = 0, 1
BM_COUNTS = ("free", "active", "cached", "host", "reused_tokens", "evictions", "offloads", "onloads", "drops")


class _TokenRange(ctypes.Structure):
    _fields_ = [("start", ctypes.c_int32), ("end", ctypes.c_int32), ("priority", ctypes.c_int32)]


class BlockManager:
    """Physical block ids for a paged cache: cross-request reuse, priority-LRU eviction
    with retention ranges, host offload.  Host bookkeeping only; see include/pkv_bm.h."""

    def __init__(self, num_blocks, block_size, host_blocks=0, offload_min_priority=35, default_priority=35):
        import numpy as np
        self._np = np
        self.num_blocks, self.block_size, self.host_blocks = num_blocks, block_size, host_blocks
        self._h = lib().pkv_bm_create(num_blocks, block_size, host_blocks, offload_min_priority, default_priority)
        if not self._h:
            raise PkvError("pkv_bm_create: invalid argument")

    def __del__(self):
        h, self._h = getattr(self, "_h", None), None
        if h and _lib is not None:
            _lib.pkv_bm_destroy(h)

    def _a(self, x, dtype):
        return self._np.ascontiguousarray(x, dtype=dtype)

    def add_sequence(self, seq_id, tokens, ranges=()):
        """Returns (block table as a list, number of reused prompt tokens)."""
        np = self._np
        toks = self._a(tokens, np.int32)
        rr = (_TokenRange * max(1, len(ranges)))(*[_TokenRange(int(a), int(b), int(c)) for a, b, c in ranges])
        cap = -(-len(toks) // self.block_size)
        table = np.empty(max(cap, 1), dtype=np.int32)
        r = lib().pkv_bm_add_sequence(self._h, int(seq_id), toks.ctypes.data, len(toks), rr, len(ranges),
                                      table.ctypes.data, cap)
        if r < 0:
            _check("bm_add_sequence", r)
        return table[:cap].tolist(), r

    def append_tokens(self, seq_ids, tokens):
        """One decode step: the cache slot of each sequence's new token (int64 array)."""
        np = self._np
        ids, toks = self._a(seq_ids, np.int64), self._a(tokens, np.int32)
        slots = np.empty(len(ids), dtype=np.int64)
        done = ctypes.c_int(0)
        r = lib().pkv_bm_append_tokens(self._h, ids.ctypes.data, toks.ctypes.data, len(ids), slots.ctypes.data,
                                       ctypes.byref(done))
        if r < 0:
            msg = lib().pkv_status_str(r).decode()
            raise PkvError(f"bm_append_tokens: {msg} after {done.value} of {len(ids)} sequences")
        return slots

    def release(self, seq_id):
        _check("bm_release", lib().pkv_bm_release(self._h, int(seq_id)))

    def slide_window(self, seq_id, window):
        r = lib().pkv_bm_slide_window(self._h, int(seq_id), int(window))
        if r < 0:
            _check("bm_slide_window", r)
        return r

    def tables(self, seq_ids, max_blocks):
        """(block tables int32 [n][max_blocks], context lengths int32 [n]) for an attention call."""
        np = self._np
        ids = self._a(seq_ids, np.int64)
        t = np.empty((len(ids), max_blocks), dtype=np.int32)
        c = np.empty(len(ids), dtype=np.int32)
        _check("bm_tables", lib().pkv_bm_tables(self._h, ids.ctypes.data, len(ids), t.ctypes.data, max_blocks,
                                                c.ctypes.data))
        return t, c

    def take_copies(self):
        """Copies recorded since the last call: int32 [n][3] rows (kind, src, dst)."""
        np = self._np
        n = lib().pkv_bm_pending_copies(self._h)
        out = np.empty((max(n, 1), 3), dtype=np.int32)
        r = lib().pkv_bm_take_copies(self._h, out.ctypes.data, n)
        if r < 0:
            _check("bm_take_copies", r)
        return out[:r]

    def counts(self):
        out = (ctypes.c_int64 * len(BM_COUNTS))()
        lib().pkv_bm_counts(self._h, out)
        return dict(zip(BM_COUNTS, list(out)))


def copy_blocks(copies, k_pool, v_pool, k_host, v_host, stream=None):
    """Apply recorded copies (int32 [n][3] rows kind, src, dst) between the device pools and
    host pools in page-locked memory ([host_blocks][...] tensors of the same block shape)."""
    import numpy as np
    _cuda(k_pool, v_pool)
    for t in (k_host, v_host):
        if t.is_cuda or not t.is_pinned() or not t.is_contiguous():
            raise PkvError("host pools must be contiguous page-locked CPU tensors")
    assert k_pool.shape[1:] == k_host.shape[1:] and k_pool.dtype == k_host.dtype
    c = np.ascontiguousarray(copies, dtype=np.int32).reshape(-1, 3)
    block_bytes = k_pool[0].numel() * k_pool.element_size()
    _check("copy_blocks", lib().pkv_copy_blocks(c.ctypes.data, len(c), _ptr(k_pool), _ptr(v_pool), k_pool.shape[0],
                                                _ptr(k_host), _ptr(v_host), k_host.shape[0], block_bytes,
                                                _stream(stream)))


# ---------------------------------------------------------------------------------------------
# CacheBlend's model-free steps (pkv.h): KV deviation, top-ratio selection, fuse.
def kv_deviation(k_pool, v_pool, slots, k_new, v_new, out=None, err=None, stream=None):
    """Per-token L2 distance between the cached K/V at slots and the recomputed rows (fp32 [n])."""
    _cuda(k_pool, v_pool, slots, k_new, v_new, out, err)
    assert k_pool.dtype == v_pool.dtype == k_new.dtype == v_new.dtype == torch.bfloat16
    assert slots.dtype == torch.int64
    num_blocks, n_kv, bs, d = k_pool.shape
    n = slots.numel()
    assert k_new.shape == v_new.shape == (n, n_kv, d)
    dev = torch.empty(n, dtype=torch.float32, device=k_pool.device) if out is None else out
    assert dev.dtype == torch.float32 and dev.numel() == n
    _check("kv_deviation", lib().pkv_kv_deviation(_ptr(k_pool), _ptr(v_pool), _ptr(slots), _ptr(k_new), _ptr(v_new),
                                                  n, num_blocks, bs, n_kv, d, _ptr(dev), _ptr(err), _stream(stream)))
    return dev


def select_top(dev, seg_offsets, counts, out=None, stream=None):
    """Per segment, the counts[s] largest deviations as ascending global indices (int32).
    seg_offsets / counts: host sequences (they size the output), or device int32 tensors
    together with a device `out` of the right size (no host work, e.g. inside a graph)."""
    import numpy as np
    _cuda(dev, out)
    assert dev.dtype == torch.float32
    if out is None:
        offs = np.ascontiguousarray(seg_offsets, dtype=np.int32)
        cnt = np.ascontiguousarray(counts, dtype=np.int32)
        assert len(offs) == len(cnt) + 1
        total = int(np.minimum(np.maximum(cnt, 0), np.maximum(np.diff(offs), 0)).sum())
        out = torch.empty(max(total, 1), dtype=torch.int32, device=dev.device)[:total]
        seg_offsets = torch.as_tensor(offs, device=dev.device)
        counts = torch.as_tensor(cnt, device=dev.device)
    _cuda(seg_offsets, counts)
    assert seg_offsets.dtype == counts.dtype == out.dtype == torch.int32
    _check("select_top", lib().pkv_select_top(_ptr(dev), _ptr(seg_offsets), _ptr(counts), counts.numel(), _ptr(out),
                                              _stream(stream)))
    return out


def kv_fuse(k_new, v_new, row_slots, rows, k_pool, v_pool, err=None, stream=None):
    """pools[row_slots[rows[j]]] = k_new / v_new[rows[j]]: the recomputed rows of the selected tokens."""
    _cuda(k_new, v_new, rows, row_slots, k_pool, v_pool, err)
    assert rows.dtype == torch.int32 and row_slots.dtype == torch.int64 and row_slots.numel() == k_new.shape[0]
    num_blocks, n_kv, bs, d = k_pool.shape
    _check("kv_fuse", lib().pkv_kv_fuse(_ptr(k_new), _ptr(v_new), _ptr(row_slots), k_new.shape[0], _ptr(rows),
                                        rows.numel(), _ptr(k_pool), _ptr(v_pool), num_blocks, bs, n_kv, d, _ptr(err),
                                        _stream(stream)))


def recompute_ratio(load_time, full_recompute_time):
    return lib().pkv_recompute_ratio(float(load_time), float(full_recompute_time))


def select_count(ratio, n):
    return lib().pkv_select_count(float(ratio), int(n))


def selftest_wait(arrive, limit_us, err, stream=None):
    """Run the bounded-wait self-test; err (device int32) gets DEV_TIMEOUT if the wait ran out."""
    _cuda(err)
    _check("selftest_wait", lib().pkv_selftest_wait(1 if arrive else 0, int(limit_us), _ptr(err), _stream(stream)))


# ---------------------------------------------------------------------------------------------
# HBM ceiling probes (pkv.h): the read-only stream and the copy the roofline is measured against.
def probe_read(buf, sink=None, stream=None):
    """Stream every byte of the CUDA tensor `buf` once (16-byte loads)."""
    _cuda(buf, sink)
    _check("probe_read", lib().pkv_probe_read(_ptr(buf), buf.numel() * buf.element_size(), _ptr(sink),
                                              _stream(stream)))


def probe_copy(src, dst, stream=None):
    """Copy the CUDA tensor `src` into `dst` (same byte size; 16-byte loads and stores)."""
    _cuda(src, dst)
    n = src.numel() * src.element_size()
    assert dst.numel() * dst.element_size() == n
    _check("probe_copy", lib().pkv_probe_copy(_ptr(src), _ptr(dst), n, _stream(stream)))
