"""Index arithmetic of the decode work partition (host-side restatement, brute-forced).

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
