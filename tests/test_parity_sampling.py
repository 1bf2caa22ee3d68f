"""Host logic of the parity tests' row sampling (no GPU): the CTA-pair token
tiling and the layout-aware choice of tokens for batches too large for the
oracle to do whole, on groupings from the oracle's own routing."""
import numpy as np

import helpers
import oracle


def test_pair_token_tiles():
    """ceil(cnt / 256) tiles of equal height rounded up to 16 rows."""
    assert helpers.pair_token_tiles(0) == []
    assert helpers.pair_token_tiles(1) == [(0, 1)]
    assert helpers.pair_token_tiles(256) == [(0, 256)]
    assert helpers.pair_token_tiles(257) == [(0, 144), (144, 113)]
    assert helpers.pair_token_tiles(1024) == [(0, 256), (256, 256), (512, 256), (768, 256)]
    for cnt in range(1, 3000, 37):
        tiles = helpers.pair_token_tiles(cnt)
        assert sum(n for _, n in tiles) == cnt
        assert all(n <= 256 for _, n in tiles)
        assert all(s % 16 == 0 for s, _ in tiles)


def _routing(T, E, k, seed, bias=None):
    rng = np.random.default_rng(seed)
    logits = rng.standard_normal((T, E)).astype(np.float32)
    if bias is not None:
        logits += np.asarray(bias, np.float32)
    idx, _, counts, offsets, perm, _ = oracle.load().route(logits, k)
    return idx, counts, offsets, perm


def test_layout_rows_cover_edges_and_every_expert():
    for T, E, k, bias in ((4096, 8, 2, None), (8192, 8, 2, (2, 1, 0, 0, 0, 0, -1, -2)),
                          (300, 5, 2, None)):
        idx, counts, offsets, perm = _routing(T, E, k, seed=T, bias=bias)
        rows = helpers.layout_rows(idx, offsets, perm, k, per_expert=16, seed=1)
        chosen = set(rows.tolist())
        assert len(chosen) == len(rows) and rows.min() >= 0 and rows.max() < T
        for e in range(E):
            lo, hi = int(offsets[e]), int(offsets[e + 1])
            if hi == lo:
                continue
            # the first and last grouped rows of the expert
            assert perm[lo] // k in chosen and perm[hi - 1] // k in chosen
            # every CTA-pair tile's first and last row
            for s0, n in helpers.pair_token_tiles(hi - lo):
                assert perm[lo + s0] // k in chosen
                assert perm[lo + s0 + n - 1] // k in chosen
            # every 128-row boundary of the one-CTA tiles
            for b in range(128, hi - lo, 128):
                assert perm[lo + b - 1] // k in chosen and perm[lo + b] // k in chosen
            assert (idx[rows] == e).any(1).sum() >= min(16, hi - lo)


def test_layout_rows_keep_required_tokens():
    idx, _, offsets, perm = _routing(500, 8, 2, seed=3)
    rows = helpers.layout_rows(idx, offsets, perm, 2, per_expert=4, must=[7, 499])
    assert 7 in rows and 499 in rows
