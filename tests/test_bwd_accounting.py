"""Host logic of the backward's measurement (CPU only).

``bench.bwd_tile_visits`` gives the 64 x 64 pair tiles each backward kernel
computes, from the kernels' loop bounds; the executed-FLOP figure that
``bench.py --bwd`` reports multiplies them by each tile's multiply-adds.  The
loop bounds are meant to visit exactly the tiles that hold at least one pair
the score keeps (query row i < L, key j < M + L, j <= M + i: "Transformer-XL:
Attentive Language Models Beyond a Fixed-Length Context", §3.2, the causal
offset over the extended context), each once.  Checked here by brute force
over every pair of small shapes: ragged rows, keys and distances, no memory,
one query, segments of one, two and several row chunks.
"""

import numpy as np
import pytest

import bench

T = 64


def _kept(L, M):
    K = M + L
    i = np.arange(L)[:, None]
    j = np.arange(K)[None, :]
    return j <= M + i  # [L, K]


def _tiles_with_pairs(mask, T=T):
    rows, cols = mask.shape
    n = 0
    for r0 in range(0, rows, T):
        for c0 in range(0, cols, T):
            n += bool(mask[r0:r0 + T, c0:c0 + T].any())
    return n


@pytest.mark.parametrize("B,H,L,M", [(1, 1, 1, 200), (2, 3, 50, 70), (1, 2, 65, 0), (2, 1, 64, 64),
                                     (1, 2, 128, 1600), (1, 1, 130, 130), (3, 2, 300, 200),
                                     (1, 1, 128, 64), (1, 1, 200, 0)])
def test_tile_visits_are_the_tiles_with_kept_pairs(B, H, L, M):
    v = bench.bwd_tile_visits(B, H, L, M)
    kept = _kept(L, M)
    # query chunk x key tile
    by_key = _tiles_with_pairs(kept)
    # query chunk x distance tile: pair (i, d) is key M + i - d
    K = M + L
    i = np.arange(L)[:, None]
    d = np.arange(K)[None, :]
    by_dist = _tiles_with_pairs((d <= M + i) & (M + i - d < K))
    assert v["stats"] == B * H * by_key
    assert v["dr"] == H * B * by_dist
    assert v["chunks"] == B * H * (-(-L // T))
    if -(-L // T) <= 2:
        assert v["dqkv"] == B * H * by_key and "dq" not in v
    else:
        assert v["dq"] == B * H * by_key and v["dkv"] == B * H * by_key and "dqkv" not in v


def test_headline_tile_counts():
    # B = 16, H = 16, L = 128, M = 1600: 27 key tiles; chunk 0's last kept key
    # is 1663, so the 27th tile (keys 1664..1727) holds pairs of chunk 1 only
    v = bench.bwd_tile_visits(16, 16, 128, 1600)
    assert v["stats"] == 256 * (26 + 27) == 13568
    assert v["dqkv"] == 13568 and v["dr"] == 13568
