"""Pins the oracle's block manager (CPU only) against the rules the page states.

"KV 캐시 시스템 (KV Cache System)": blocks are reusable across requests until evicted;
eviction is priority-based LRU with priorities 0..100 (lower freed first); retention
token ranges set priorities; blocks below secondary_offload_min_priority (35) are
evicted without offload, others go to host memory and come back on reuse; blocks that
leave the attention window are released into the tree.  Plus invariants on random
traces and an end-to-end data check through the recorded copies.
"""
import numpy as np
import pytest

import oracle
from oracle.block_manager import OFFLOAD, ONLOAD


def _toks(base, n):
    return [base * 1000 + i for i in range(n)]


def test_reuse_across_requests_until_evicted():
    bm = oracle.BlockManager(8, 4)
    t1, r1 = bm.add_sequence(1, _toks(1, 10))
    assert r1 == 0 and len(t1) == 3
    bm.release(1)
    t2, r2 = bm.add_sequence(2, _toks(1, 10))             # same prompt: two full blocks reused
    assert r2 == 8 and t2[:2] == t1[:2]
    t3, r3 = bm.add_sequence(3, _toks(1, 9) + [7])        # shares the first two blocks, in use
    assert r3 == 8 and t3[:2] == t1[:2]
    assert bm.gpu_ref[t1[0]] == 2
    bm.release(2); bm.release(3)
    # fill the pool with other requests: the cached blocks get evicted, reuse is gone
    bm.add_sequence(4, _toks(4, 32))
    bm.release(4)
    t6, r6 = bm.add_sequence(6, _toks(1, 10))
    assert r6 == 0


def test_lower_priority_is_evicted_first():
    bm = oracle.BlockManager(5, 4)
    bm.add_sequence(1, _toks(1, 8), ranges=[(0, -1, 80)])   # 2 full blocks, priority 80
    bm.add_sequence(2, _toks(2, 8), ranges=[(0, -1, 20)])   # 2 full blocks, priority 20
    bm.release(2)                                            # released first: older
    bm.release(1)
    t, _ = bm.add_sequence(3, _toks(3, 8))                   # needs 2 blocks: evicts both of seq 2
    assert bm.add_sequence(4, _toks(1, 9))[1] == 8           # seq 1's blocks survived
    assert bm.stats["evictions"] == 2


def test_lru_within_one_priority():
    bm = oracle.BlockManager(5, 4)
    bm.add_sequence(1, _toks(1, 8))
    bm.add_sequence(2, _toks(2, 8))
    bm.release(1)                                            # older
    bm.release(2)
    bm.add_sequence(3, _toks(3, 8))                          # evicts seq 1's blocks
    assert bm.add_sequence(4, _toks(2, 9))[1] == 8
    bm.release(4)
    assert bm.add_sequence(5, _toks(1, 9))[1] == 0


def test_retention_range_example():
    # "tokens 10 to 61 get priority X": with 16-token blocks, blocks 0..3 overlap [10, 61)
    bm = oracle.BlockManager(16, 16, default_priority=35)
    bm.add_sequence(1, list(range(100)), ranges=[(10, 61, 90)])
    pr = bm.seqs[1]["prios"]
    assert pr == [90, 90, 90, 90, 35, 35, 35]
    # overlapping ranges: the highest wins; an open range covers decode tokens too
    bm.add_sequence(2, list(range(200, 240)), ranges=[(0, 20, 10), (16, 17, 60), (32, -1, 5)])
    assert bm.seqs[2]["prios"] == [10, 60, 5]
    for t in range(9):
        bm.append_token(2, 999)
    assert bm.seqs[2]["prios"] == [10, 60, 5, 5]


def test_offload_threshold():
    # below 35: evicted without offload; at 35: offloaded, and reused through an onload
    bm = oracle.BlockManager(2, 4, host_blocks=4, offload_min_priority=35)
    bm.add_sequence(1, _toks(1, 5), ranges=[(0, -1, 34)])
    bm.release(1)
    bm.add_sequence(2, _toks(2, 5))
    assert bm.take_copies() == [] and bm.counts()["host"] == 0
    bm.release(2)
    bm.add_sequence(3, _toks(3, 5))                          # evicts seq 2's full block (35)
    c = bm.take_copies()
    assert [k for k, _, _ in c] == [OFFLOAD] and bm.counts()["host"] == 1
    bm.release(3)
    t4, r4 = bm.add_sequence(4, _toks(2, 5))                 # seq 2's block comes back
    c = bm.take_copies()
    assert r4 == 4 and ONLOAD in [k for k, _, _ in c]
    assert bm.stats["onloads"] == 1


def test_host_eviction_is_priority_lru():
    bm = oracle.BlockManager(2, 2, host_blocks=2)
    for sid, prio in [(1, 50), (2, 40), (3, 60)]:
        bm.add_sequence(sid, _toks(sid, 3), ranges=[(0, -1, prio)])
        bm.release(sid)
        # two GPU blocks, one full + one partial per request: each new request pushes the
        # previous request's full block out to the host
    # host now held seq 1 (50) and seq 2 (40); seq 3's block is cached on the GPU
    bm.add_sequence(4, _toks(4, 3))                          # offloads seq 3's block: host evicts 40
    bm.release(4)
    hosts = sorted(bm.nodes[n]["prio"] for n in bm.host_node if n is not None)
    assert hosts == [50, 60]


def test_at_least_one_token_is_computed():
    bm = oracle.BlockManager(8, 4)
    bm.add_sequence(1, _toks(1, 8))
    bm.release(1)
    assert bm.add_sequence(2, _toks(1, 8))[1] == 4           # 2 full blocks match, 1 reused
    assert bm.add_sequence(3, _toks(1, 9))[1] == 8


def test_window_releases_blocks_into_the_tree():
    bm = oracle.BlockManager(16, 4)
    bm.add_sequence(1, _toks(1, 20))
    first = bm.slide_window(1, 6)                            # tokens 14..19 stay: blocks 3, 4
    assert first == 3
    assert bm.counts()["cached"] == 3 and bm.counts()["active"] == 2
    assert bm.add_sequence(2, _toks(1, 13))[1] == 12         # the released prefix is reused


def _content(tokens, pos):
    return tokens[pos] * 7 + pos


@pytest.mark.parametrize("seed", [0, 1, 2, 3])
def test_random_traces_keep_invariants_and_data(seed):
    """Random requests over a few shared prefixes on a small pool with a host tier.  KV
    content is a function of (token, position), written at every computed slot; after
    applying the recorded copies, every sequence's cache must hold its own content."""
    rng = np.random.default_rng(seed)
    N, bs, H = 24, 4, 10
    bm = oracle.BlockManager(N, bs, host_blocks=H)
    gpu = np.full((N, bs), -1, dtype=np.int64)
    host = np.full((H, bs), -1, dtype=np.int64)
    prefixes = [list(rng.integers(0, 50, size=int(rng.integers(4, 14)))) for _ in range(4)]
    live = {}
    sid = 0
    for step in range(300):
        op = rng.random()
        if op < 0.35 or not live:
            sid += 1
            toks = list(prefixes[int(rng.integers(0, 4))]) + list(rng.integers(0, 50, size=int(rng.integers(1, 6))))
            prio = int(rng.integers(0, 101))
            try:
                table, reused = bm.add_sequence(sid, toks, ranges=[(0, int(rng.integers(1, 12)), prio)])
            except oracle.OutOfBlocks:
                oracle.apply_copies(bm.take_copies(), gpu, host)
                continue
            oracle.apply_copies(bm.take_copies(), gpu, host)
            for pos in range(reused, len(toks)):             # the prefill writes the rest
                gpu[table[pos // bs], pos % bs] = _content(toks, pos)
            live[sid] = toks
        elif op < 0.75:
            s = list(live)[int(rng.integers(0, len(live)))]
            tok = int(rng.integers(0, 50))
            try:
                slot = bm.append_token(s, tok)
            except oracle.OutOfBlocks:
                oracle.apply_copies(bm.take_copies(), gpu, host)
                continue
            oracle.apply_copies(bm.take_copies(), gpu, host)
            live[s].append(tok)
            gpu[slot // bs, slot % bs] = _content(live[s], len(live[s]) - 1)
        elif op < 0.9:
            s = list(live)[int(rng.integers(0, len(live)))]
            bm.release(s)
            del live[s]
        else:
            s = list(live)[int(rng.integers(0, len(live)))]
            bm.slide_window(s, int(rng.integers(1, 12)))
        # invariants
        c = bm.counts()
        assert c["free"] + c["active"] + c["cached"] == N
        refs = np.zeros(N, int)
        for s, seq in bm.seqs.items():
            for b in seq["blocks"][seq["first"]:]:
                refs[b] += 1
        assert list(refs) == bm.gpu_ref
        for nid, n in bm.nodes.items():
            assert bm.index[(n["parent"], n["key"])] == nid
            kind, where = n["loc"]
            assert (bm.gpu_node if kind == "gpu" else bm.host_node)[where] == nid
        # data: every held position of every live sequence holds its own content
        for s, toks in live.items():
            seq = bm.seqs[s]
            for pos in range(seq["first"] * bs, len(toks)):
                assert gpu[seq["blocks"][pos // bs], pos % bs] == _content(toks, pos), (seed, step, s, pos)


def test_planted_mistake_highest_priority_first_is_caught():
    # a manager that evicts the highest priority first fails the priority pin
    class Wrong(oracle.BlockManager):
        def _evict_one(self):
            cands = [(-self.nodes[self.gpu_node[b]]["prio"], self.nodes[self.gpu_node[b]]["time"],
                      -self.nodes[self.gpu_node[b]]["depth"], b) for b in range(self.N) if self._gpu_state(b) == "cached"]
            if not cands:
                raise oracle.OutOfBlocks()
            b = min(cands)[3]
            self._drop(self.gpu_node[b])
    bm = Wrong(5, 4)
    bm.add_sequence(1, _toks(1, 8), ranges=[(0, -1, 80)])
    bm.add_sequence(2, _toks(2, 8), ranges=[(0, -1, 20)])
    bm.release(2); bm.release(1)
    bm.add_sequence(3, _toks(3, 8))
    assert bm.add_sequence(4, _toks(1, 9))[1] != 8
