"""The paged-layout generator (synth/paging.py), on the CPU: every key of
every sequence lands on exactly one physical row of a page its table row
names, and nothing else is claimed."""

import numpy as np
import pytest

from synth.paging import page_layout


@pytest.mark.parametrize("P", [32, 128])
def test_every_key_has_one_row_and_the_table_covers_it(P):
    rng = np.random.default_rng(3)
    ctx = rng.integers(1, 700, size=9)
    M = 3
    rs = np.concatenate([[0], np.cumsum(ctx + M - 1 + 2)[:-1]])   # gaps between sequences
    L = page_layout(ctx, rs, M, P, seed=5)
    seen = []
    for b in range(len(ctx)):
        n = ctx[b] + M - 1
        used = (n + P - 1) // P
        assert (L.block_table[b, :used] >= 0).all() and (L.block_table[b, used:] == -1).all()
        t = np.arange(n)
        phys = L.block_table[b, t // P].astype(np.int64) * P + t % P
        assert np.array_equal(L.src[phys], rs[b] + t)
        seen.append(phys)
    seen = np.concatenate(seen)
    assert len(np.unique(seen)) == len(seen)                      # no two keys share a row
    assert (L.src >= 0).sum() == len(seen)                        # no other row is claimed
    assert L.block_table.max() < L.n_pages
    pages = L.block_table[L.block_table >= 0]
    assert len(np.unique(pages)) == len(pages)                    # no page is shared
