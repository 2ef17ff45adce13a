"""The native block manager (include/pkv_bm.h) against the oracle's BlockManager on
seeded random request traces: identical block tables, reused-token counts, slots,
recorded copies, failures and counters at every step.  Host code only (no GPU)."""
import numpy as np
import pytest

import oracle
import paged_kv_cache_175_gb300 as pkv


def _run_trace(seed, N, bs, H, steps, offload_min=35, n_prefix=4, window_ops=True):
    rng = np.random.default_rng(seed)
    ref = oracle.BlockManager(N, bs, host_blocks=H, offload_min_priority=offload_min)
    nat = pkv.BlockManager(N, bs, host_blocks=H, offload_min_priority=offload_min)
    prefixes = [list(rng.integers(0, 40, size=int(rng.integers(bs, 4 * bs)))) for _ in range(n_prefix)]
    live = []
    sid = 0
    for step in range(steps):
        op = rng.random()
        if op < 0.3 or not live:
            sid += 1
            toks = list(prefixes[int(rng.integers(0, n_prefix))]) + list(rng.integers(0, 40, size=int(rng.integers(1, 2 * bs))))
            ranges = [(int(rng.integers(0, 8)), int(rng.integers(-1, 30)), int(rng.integers(0, 101)))
                      for _ in range(int(rng.integers(0, 3)))]
            try:
                want = ref.add_sequence(sid, toks, ranges=ranges)
            except oracle.OutOfBlocks:
                want = None
            try:
                got = nat.add_sequence(sid, toks, ranges=ranges)
            except pkv.PkvError:
                got = None
            assert got == want, (seed, step)
            if want is not None:
                live.append(sid)
        elif op < 0.7:
            batch = [live[int(i)] for i in rng.choice(len(live), size=min(len(live), int(rng.integers(1, 5))), replace=False)]
            toks = [int(t) for t in rng.integers(0, 40, size=len(batch))]
            want, fail_ref = [], False
            for s, t in zip(batch, toks):
                try:
                    want.append(ref.append_token(s, t))
                except oracle.OutOfBlocks:
                    fail_ref = True
                    break
            try:
                got = list(nat.append_tokens(batch, toks))
                fail_nat = False
            except pkv.PkvError as e:
                fail_nat = True
                assert f"after {len(want)} of" in str(e), (str(e), len(want))
            assert fail_nat == fail_ref, (seed, step)
            if not fail_nat:
                assert got == want, (seed, step)
        elif op < 0.88 or not window_ops:
            s = live.pop(int(rng.integers(0, len(live))))
            ref.release(s)
            nat.release(s)
        else:
            s = live[int(rng.integers(0, len(live)))]
            w = int(rng.integers(1, 3 * bs))
            assert nat.slide_window(s, w) == ref.slide_window(s, w)
        want_c = [list(c) for c in ref.take_copies()]
        got_c = nat.take_copies().tolist()
        assert got_c == want_c, (seed, step)
        c = nat.counts()
        rc = ref.counts()
        assert (c["free"], c["active"], c["cached"], c["host"]) == (rc["free"], rc["active"], rc["cached"], rc["host"]), (seed, step)
        for k in ("reused_tokens", "evictions", "offloads", "onloads", "drops"):
            assert c[k] == ref.stats[k], (seed, step, k)
        if live and step % 7 == 0:
            mb = max(len(ref.seqs[s]["blocks"]) for s in live)
            t, ctx = nat.tables(live, mb + 1)
            for r, s in enumerate(live):
                blocks, n = ref.table(s)
                first = ref.seqs[s]["first"]
                exp = [-1] * first + blocks[first:] + [-1] * (mb + 1 - len(blocks))
                assert t[r].tolist() == exp and ctx[r] == n
    return ref.stats


@pytest.mark.parametrize("seed", range(6))
def test_native_matches_oracle_with_host_tier(seed):
    st = _run_trace(seed, N=32, bs=4, H=12, steps=400)
    assert st["offloads"] > 0 and st["evictions"] > 0


@pytest.mark.parametrize("seed", range(3))
def test_native_matches_oracle_without_host_tier(seed):
    _run_trace(100 + seed, N=20, bs=2, H=0, steps=300)


def test_native_matches_oracle_block16():
    st = _run_trace(7, N=64, bs=16, H=64, steps=800, n_prefix=6)
    assert st["reused_tokens"] > 0 and st["onloads"] > 0 and st["drops"] > 0


def test_offload_threshold_zero_and_above_max():
    # threshold 0: every victim goes to the host; 101: none does
    for thr, expect in ((0, True), (101, False)):
        nat = pkv.BlockManager(2, 2, host_blocks=4, offload_min_priority=thr)
        for s in range(1, 5):
            nat.add_sequence(s, [s * 10, s * 10 + 1, s * 10 + 2], ranges=[(0, -1, 0)])
            nat.release(s)
        assert (nat.counts()["offloads"] > 0) == expect


def test_bad_arguments():
    with pytest.raises(pkv.PkvError):
        pkv.BlockManager(0, 16)
    nat = pkv.BlockManager(4, 4)
    nat.add_sequence(1, [1, 2, 3])
    with pytest.raises(pkv.PkvError):
        nat.add_sequence(1, [1, 2, 3])                   # duplicate id
    with pytest.raises(pkv.PkvError):
        nat.release(2)                                    # unknown id
    with pytest.raises(pkv.PkvError):
        nat.add_sequence(3, [1], ranges=[(0, 4, 101)])    # priority out of range
    with pytest.raises(pkv.PkvError):
        nat.tables([1], 0)                                # table too small
