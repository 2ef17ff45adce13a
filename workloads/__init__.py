"""Seeded synthetic inputs for the paged decode path.

This module is shared by the oracle side and the CUDA side of the tests and of
the benchmark.  It holds no arithmetic of the method itself: it draws context
lengths, hands out physical block ids the way a block manager would (a seeded
permutation of a shared pool, optionally with a shared prefix), and draws the
q / K / V values.  Everything is reproducible from ``seed``.

Workloads (shapes of the decode layers the reference pages talk about):

* ``tiny``        1 layer, batch 4, ctx {17, 64, 100, 255}, 8 q / 2 kv heads,
                  head_dim 64, block 16, pool of 128 blocks.
* ``llama3_8b``   32 q / 8 kv heads, head_dim 128, block 16, batch 64,
                  ctx ~ U[512, 4096], pool = 1.2 x the blocks needed.
* ``llama2_70b_prefix``  64 q / 8 kv heads, head_dim 128, block 16, batch 128,
                  ctx lognormal(median 2048, sigma 0.6) clipped to [256, 8192];
                  the first 32 sequences share one 2048-token prefix
                  (the same 128 physical blocks).
* ``mqa_bs16`` / ``mqa_bs32`` / ``mha_bs16`` / ``mha_bs32``  32 q heads,
                  n_kv = 1 (MQA) or 32 (MHA), head_dim 128, batch 256, ctx 2048.
* ``int4_long``   32 q / 8 kv heads, head_dim 128, batch 32, ctx ~ U[8192, 32768],
                  K with 4 outlier channels per kv head (std 10), block 16
                  (``int4_long_bs64``: block 64).
* ``<name>_window<W>``  the named workload for a layer with a limited attention
                  window of W tokens (e.g. ``llama3_8b_window256``: the 256-token
                  layers of a max_attention_window = [4096, 256] model).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch


@dataclass
class Workload:
    name: str
    batch: int
    n_h: int
    n_kv: int
    head_dim: int
    block_size: int
    context_lens: np.ndarray          # int32 [batch]; includes the token appended this step
    block_tables: np.ndarray          # int32 [batch][max_blocks]; unused entries are -1
    num_blocks: int                   # size of the shared physical pool
    scale: float
    shared_prefix_blocks: int = 0     # number of leading table entries shared by the sharers
    n_sharers: int = 0
    outlier_channels: np.ndarray | None = None   # int [n_kv][4] (int4 workload only)
    extra: dict = field(default_factory=dict)
    window: int = 0                   # attention window in tokens (0: whole context)

    @property
    def group(self) -> int:
        return self.n_h // self.n_kv

    @property
    def max_blocks(self) -> int:
        return self.block_tables.shape[1]

    def blocks_of(self, s: int) -> int:
        return -(-int(self.context_lens[s]) // self.block_size)

    def unique_blocks(self) -> int:
        used = set()
        for s in range(self.batch):
            used.update(self.block_tables[s, : self.blocks_of(s)].tolist())
        return len(used)


def _tables(ctx: np.ndarray, bs: int, rng: np.random.Generator, pool_factor: float,
            pool_blocks: int | None = None, shared: int = 0, n_sharers: int = 0):
    """Assign physical blocks from a shuffled pool, as a block manager would.

    Sequences ``0 .. n_sharers-1`` reuse the same ``shared`` leading blocks.
    """
    nb = [-(-int(c) // bs) for c in ctx]
    private = [n - (shared if s < n_sharers else 0) for s, n in enumerate(nb)]
    need = sum(private) + (shared if n_sharers else 0)
    num_blocks = pool_blocks if pool_blocks is not None else int(math.ceil(pool_factor * need))
    assert num_blocks >= need
    perm = rng.permutation(num_blocks).astype(np.int32)
    max_blocks = max(nb)
    bt = np.full((len(ctx), max_blocks), -1, dtype=np.int32)
    cur = 0
    prefix = None
    if n_sharers:
        prefix = perm[cur: cur + shared]
        cur += shared
    for s, n in enumerate(nb):
        if s < n_sharers:
            bt[s, :shared] = prefix
            bt[s, shared:n] = perm[cur: cur + n - shared]
            cur += n - shared
        else:
            bt[s, :n] = perm[cur: cur + n]
            cur += n
    return bt, num_blocks


def make(name: str, seed: int = 0) -> Workload:
    """Shapes, context lengths and block tables of a named workload (host only).

    A suffix ``_b<N>`` keeps the first N context lengths of the named workload with a
    pool sized for them (a smaller case of the same shape, e.g. for profiler captures).
    """
    wbase, _, wv = name.rpartition("_window")
    if wbase and wv.isdigit():
        w = make(wbase, seed)
        w.name, w.window = name, int(wv)
        return w
    base, _, nb = name.rpartition("_b")
    if base and nb.isdigit() and base in NAMES:
        w = make(base, seed)
        n = int(nb)
        ctx = w.context_lens[:n].copy()
        bt, nbk = _tables(ctx, w.block_size, np.random.default_rng(seed + 1), 1.2,
                          shared=w.shared_prefix_blocks, n_sharers=min(w.n_sharers, n))
        return Workload(name, n, w.n_h, w.n_kv, w.head_dim, w.block_size, ctx, bt, nbk, w.scale,
                        shared_prefix_blocks=w.shared_prefix_blocks if min(w.n_sharers, n) else 0,
                        n_sharers=min(w.n_sharers, n), outlier_channels=w.outlier_channels, extra=w.extra)
    rng = np.random.default_rng(seed)
    if name == "tiny":
        ctx = np.array([17, 64, 100, 255], dtype=np.int32)
        bt, nbk = _tables(ctx, 16, rng, 1.0, pool_blocks=128)
        return Workload(name, 4, 8, 2, 64, 16, ctx, bt, nbk, 1.0 / math.sqrt(64))
    if name == "llama3_8b":
        ctx = rng.integers(512, 4097, size=64).astype(np.int32)
        bt, nbk = _tables(ctx, 16, rng, 1.2)
        return Workload(name, 64, 32, 8, 128, 16, ctx, bt, nbk, 1.0 / math.sqrt(128))
    if name == "llama2_70b_prefix":
        raw = np.rint(rng.lognormal(mean=math.log(2048.0), sigma=0.6, size=128))
        ctx = np.clip(raw, 256, 8192).astype(np.int32)
        ctx[:32] = np.maximum(ctx[:32], 2064)       # each sharer keeps >= 1 private block
        bt, nbk = _tables(ctx, 16, rng, 1.2, shared=128, n_sharers=32)
        return Workload(name, 128, 64, 8, 128, 16, ctx, bt, nbk, 1.0 / math.sqrt(128),
                        shared_prefix_blocks=128, n_sharers=32)
    if name.startswith("mqa_") or name.startswith("mha_"):
        bs = int(name.split("bs")[1])
        n_kv = 1 if name.startswith("mqa") else 32
        ctx = np.full(256, 2048, dtype=np.int32)
        bt, nbk = _tables(ctx, bs, rng, 1.2)
        w = Workload(name, 256, 32, n_kv, 128, bs, ctx, bt, nbk, 1.0 / math.sqrt(128))
        # chunk reuse: 64 chunks of 512 tokens (the first 512 tokens of sequences 0..63),
        # each re-positioned by a seeded delta in [0, 8192]
        per_chunk = 512 // bs
        deltas = rng.integers(0, 8193, size=64).astype(np.int32)
        w.extra["rope_block_ids"] = np.concatenate([bt[c, :per_chunk] for c in range(64)]).astype(np.int32)
        w.extra["rope_deltas"] = np.repeat(deltas, per_chunk).astype(np.int32)
        return w
    if name in ("int4_long", "int4_long_bs64"):
        bs = 64 if name.endswith("bs64") else 16
        ctx = rng.integers(8192, 32769, size=32).astype(np.int32)
        bt, nbk = _tables(ctx, bs, rng, 1.2)
        outl = np.stack([rng.choice(128, size=4, replace=False) for _ in range(8)]).astype(np.int64)
        return Workload(name, 32, 32, 8, 128, bs, ctx, bt, nbk, 1.0 / math.sqrt(128),
                        outlier_channels=outl)
    raise KeyError(name)


NAMES = ["tiny", "llama3_8b", "llama2_70b_prefix", "mqa_bs16", "mqa_bs32", "mha_bs16",
         "mha_bs32", "int4_long", "int4_long_bs64"]


def generator(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def normal_bf16(shape, seed: int, device="cpu", std: float = 1.0) -> torch.Tensor:
    """N(0, std^2) draws in fp32, stored as bf16 (torch's round-to-nearest-even)."""
    x = torch.randn(*shape, generator=generator(seed, device), device=device, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x.to(torch.bfloat16)


def pools_bf16(w: Workload, seed: int, device="cpu"):
    """Random K and V pools [num_blocks][n_kv][block_size][head_dim] (the cache before the step)."""
    shape = (w.num_blocks, w.n_kv, w.block_size, w.head_dim)
    return normal_bf16(shape, seed * 7 + 1, device), normal_bf16(shape, seed * 7 + 2, device)


def queries(w: Workload, seed: int, device="cpu") -> torch.Tensor:
    return normal_bf16((w.batch, w.n_h, w.head_dim), seed * 7 + 3, device)


def new_tokens(w: Workload, seed: int, device="cpu"):
    """K / V of the token each sequence appends this step: [batch][n_kv][head_dim]."""
    shape = (w.batch, w.n_kv, w.head_dim)
    return normal_bf16(shape, seed * 7 + 4, device), normal_bf16(shape, seed * 7 + 5, device)


def decode_slots(w: Workload) -> np.ndarray:
    """Slot of each sequence's newest token (position ctx-1), as the block manager hands it out.

    slot = physical block id * block_size + offset in block; int64 [batch].
    """
    pos = w.context_lens.astype(np.int64) - 1
    phys = w.block_tables[np.arange(w.batch), pos // w.block_size].astype(np.int64)
    return phys * w.block_size + pos % w.block_size


def history_slots(w: Workload, s: int) -> np.ndarray:
    """Slots of every position 0..ctx-1 of sequence s, in logical order (int64)."""
    pos = np.arange(int(w.context_lens[s]), dtype=np.int64)
    phys = w.block_tables[s, pos // w.block_size].astype(np.int64)
    return phys * w.block_size + pos % w.block_size


def history_kv(w: Workload, s: int, seed: int, device="cpu"):
    """K / V history of sequence s: [ctx][n_kv][head_dim] bf16.

    K carries the workload's outlier channels (std 10) when it has them.
    """
    n = int(w.context_lens[s])
    k = torch.randn(n, w.n_kv, w.head_dim, generator=generator(seed * 1009 + 2 * s, device),
                    device=device, dtype=torch.float32)
    if w.outlier_channels is not None:
        for g in range(w.n_kv):
            k[:, g, torch.as_tensor(w.outlier_channels[g], device=device)] *= 10.0
    v = torch.randn(n, w.n_kv, w.head_dim, generator=generator(seed * 1009 + 2 * s + 1, device),
                    device=device, dtype=torch.float32)
    return k.to(torch.bfloat16), v.to(torch.bfloat16)
