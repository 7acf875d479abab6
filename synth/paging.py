"""Paged cache layouts: a block table that scatters every sequence's keys
over fixed-size pages in a seeded random order.

Like the rest of this package it only decides where rows live; it computes
nothing of the method.  A paged cache built from a contiguous one holds the
same rows, so a decode over it must return the same bytes.
"""

from dataclasses import dataclass

import numpy as np


@dataclass
class PageLayout:
    page_rows: int
    n_pages: int             # pages in the pool (cap_rows = n_pages * page_rows)
    block_table: np.ndarray  # int32 [B][max_pages]; entries past a sequence's last page are -1
    src: np.ndarray          # int64 [n_pages * page_rows]: the contiguous row now at this
                             # physical row, -1 where no key lives


def page_layout(ctx, row_start, M: int, page_rows: int, seed: int = 0, spare_pages: int = 3,
                slack_entries: int = 1) -> PageLayout:
    """Key t < ctx[b] + M - 1 of sequence b goes to page block_table[b][t // P],
    row t % P of that page; pages are a random permutation of the pool, with
    `spare_pages` pages no sequence uses and `slack_entries` unused table
    columns (filled with -1: a decode must never read them)."""
    P = int(page_rows)
    ctx = np.asarray(ctx, np.int64)
    rs = np.asarray(row_start, np.int64)
    n = ctx + (M - 1)
    pages = (n + P - 1) // P
    total = int(pages.sum()) + int(spare_pages)
    perm = np.random.default_rng(seed).permutation(total).astype(np.int64)
    bt = np.full((len(ctx), int(pages.max()) + int(slack_entries)), -1, np.int32)
    src = np.full(total * P, -1, np.int64)
    first = np.concatenate([[0], np.cumsum(pages)[:-1]])
    for b in range(len(ctx)):
        pg = perm[first[b]:first[b] + pages[b]]
        bt[b, :pages[b]] = pg
        keys = np.arange(n[b])
        src[pg[keys // P] * P + keys % P] = rs[b] + keys
    return PageLayout(page_rows=P, n_pages=total, block_table=bt, src=src)


def paged_copy(layout: PageLayout, k8, ks, v8, vs, seed: int = 0):
    """The cache arrays (torch, [Hkv][rows][d] int8 and [Hkv][rows] f32) laid
    out as `layout` says.  Rows that hold no key get finite random bytes, so
    a read of one shows up in the output."""
    import torch
    dev = k8.device
    Hkv, _, d = k8.shape
    rows = layout.n_pages * layout.page_rows
    g = torch.Generator(device=dev)
    g.manual_seed(1000003 + seed)
    kp = torch.randint(-127, 128, (Hkv, rows, d), generator=g, device=dev, dtype=torch.int8)
    vp = torch.randint(-127, 128, (Hkv, rows, d), generator=g, device=dev, dtype=torch.int8)
    ksp = torch.rand((Hkv, rows), generator=g, device=dev) + 0.5
    vsp = torch.rand((Hkv, rows), generator=g, device=dev) + 0.5
    src = torch.from_numpy(layout.src).to(dev)
    live = torch.nonzero(src >= 0).squeeze(1)
    from_rows = src[live]
    kp[:, live] = k8[:, from_rows]
    vp[:, live] = v8[:, from_rows]
    ksp[:, live] = ks[:, from_rows]
    vsp[:, live] = vs[:, from_rows]
    return kp, ksp, vp, vsp
