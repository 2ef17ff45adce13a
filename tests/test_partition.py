"""Index arithmetic of the decode work partition (host-side restatement, brute-forced),
and the producer's walk over a piece in stages of one or two blocks.

The kernels cut a line of W (sequence, kv head, block) positions into P pieces,
piece p = [floor(pW/P), floor((p+1)W/P)); a segment cut by pieces leaves one state per
non-empty piece at part index (segment + piece).  These checks pin the formulas the
CUDA code uses: the piece holding a position, the walk over the non-empty pieces of a
segment, and the uniqueness / bound of part indices, including W < P (empty pieces).
"""
import numpy as np
import pytest


def piece_of(pos, W, P):
    return ((pos + 1) * P - 1) // W


def bounds(p, W, P):
    return W * p // P, W * (p + 1) // P


def effective_pieces(W, P, min_piece=8):
    return max(1, min(P, -(-W // min_piece)))


@pytest.mark.parametrize("W,P", [(10, 4), (20, 608), (58, 608), (75000, 608), (7, 7), (1, 152), (999, 1000)])
def test_piece_of_matches_brute_force(W, P):
    owner = np.full(W, -1)
    for p in range(P):
        a, b = bounds(p, W, P)
        owner[a:b] = p
    assert (owner >= 0).all()
    for pos in range(W):
        assert piece_of(pos, W, P) == owner[pos]


@pytest.mark.parametrize("seed", range(6))
def test_segment_walk_and_part_indices(seed):
    rng = np.random.default_rng(seed)
    B, n_kv = int(rng.integers(1, 40)), int(rng.integers(1, 9))
    nb = rng.integers(0, 12, size=B)
    nb[rng.random(B) < 0.2] = 0
    cum = np.concatenate([[0], np.cumsum(nb)])
    W = int(n_kv * cum[-1])
    if W == 0:
        return
    P = int(rng.choice([3, 50, 608, W, 2 * W + 1]))
    if seed % 2:
        P = effective_pieces(W, P)          # the kernels cap the grid at ceil(W / 8) pieces
        assert all(bounds(p, W, P)[1] > bounds(p, W, P)[0] for p in range(P))   # no empty piece
    parts = set()
    for s in range(B):
        for g in range(n_kv):
            if nb[s] == 0:
                continue
            start = n_kv * cum[s] + g * nb[s]
            end = start + nb[s]
            brute = [p for p in range(P) if bounds(p, W, P)[0] < end and bounds(p, W, P)[1] > start
                     and bounds(p, W, P)[0] < bounds(p, W, P)[1]]
            p0, p1 = piece_of(start, W, P), piece_of(end - 1, W, P)
            walk, p = [], p0
            while True:                       # the reduce kernel's walk
                walk.append(p)
                if p == p1:
                    break
                p = piece_of(W * (p + 1) // P, W, P)
            assert walk == brute
            for p in walk:
                part = s * n_kv + g + p
                assert part not in parts and part < B * n_kv + P
                parts.add(part)


def stages_of_piece(nb, n_kv, p, P, pair):
    """The producer's walk over piece p, restated: stages of one block, or with `pair` of two
    consecutive blocks of one segment while the piece holds them.  Returns, per stage,
    (segment, first block, number of blocks)."""
    segs = [(s, g) for s in range(len(nb)) for g in range(n_kv) if nb[s] > 0]
    starts, pos = [], 0
    for s, g in segs:
        starts.append(pos)
        pos += nb[s]
    W = pos
    a, b = bounds(p, W, P)
    out, j = [], a
    while j < b:
        k = max(i for i, st in enumerate(starts) if st <= j)         # segment holding position j
        blk = j - starts[k]
        n = 2 if pair and blk + 1 < nb[segs[k][0]] and j + 1 < b else 1
        out.append((k, blk, n))
        j += n
    return out, segs


@pytest.mark.parametrize("seed", range(8))
def test_paired_stages_cover_each_block_once_inside_one_segment(seed):
    rng = np.random.default_rng(100 + seed)
    B, n_kv = int(rng.integers(1, 30)), int(rng.integers(1, 5))
    nb = rng.integers(0, 20, size=B)
    W = int(n_kv * nb.sum())
    if W == 0:
        return
    P = effective_pieces(W, int(rng.choice([7, 64, 608])))
    seen = []
    for p in range(P):
        stages, segs = stages_of_piece(nb, n_kv, p, P, pair=True)
        for i, (k, blk, n) in enumerate(stages):
            last = nb[segs[k][0]] - 1
            # a stage stays inside one segment, so a segment's first block opens a stage and
            # its last (possibly unfinished) block closes one
            assert blk + n - 1 <= last
            # pairs are taken whenever the segment and the piece both hold the next block
            assert not (n == 1 and blk < last and i + 1 < len(stages)), (p, i, k, blk)
            seen.extend((k, blk + d) for d in range(n))
    expected = [(k, i) for k, (s, g) in enumerate(segs) for i in range(nb[s])]
    assert sorted(seen) == expected                                      # every block exactly once
