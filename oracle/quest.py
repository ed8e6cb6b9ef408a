"""Quest page metadata and query-dependent page selection (oracle; test infra).

SparseEngine "What it is" / "How it works": Quest selects pages per query at
decode time (build_decode_selection) and keeps the full KV history resident
("How it differs").  The bound is fixed by the workload text: for page p and
KV group g,

    U_g(p) = sum_{h in g} sum_i max(q_{h,i} * kmax_{p,i}, q_{h,i} * kmin_{p,i})

with kmin / kmax the elementwise min / max of the page's resident keys.
Top ``top_pages`` full pages by (U desc, block asc) plus the current (last)
page.  reading (x): the group's heads are summed (not maxed); 1/sqrt(d) is left
out since it does not change the ranking.
"""
from __future__ import annotations

import numpy as np

from .cache import Cache, cdiv, values
from .selection import rank


def page_minmax(c: Cache, b: int, h: int, block: int):
    """Elementwise (min, max) over the resident keys of one block, as raw bits
    of the same dtype (min / max of representable values is exact)."""
    P = c.page_size
    ctx = int(c.ctx_len[b])
    rows = min(P, ctx - block * P)
    page = int(c.block_table[b, block])
    kv = values(c.k[page, h, :rows, :])
    kmin, kmax = kv.min(axis=0), kv.max(axis=0)
    return kmin, kmax


def build_meta(c: Cache, seqs=None):
    """kmin, kmax as fp64 arrays indexed [page][Hkv][D] (pages of ``seqs``)."""
    num_pages = c.k.shape[0]
    kmin = np.zeros((num_pages, c.Hkv, c.D))
    kmax = np.zeros((num_pages, c.Hkv, c.D))
    for b in (range(c.B) if seqs is None else seqs):
        for blk in range(cdiv(int(c.ctx_len[b]), c.page_size)):
            page = int(c.block_table[b, blk])
            for h in range(c.Hkv):
                kmin[page, h], kmax[page, h] = page_minmax(c, b, h, blk)
    return kmin, kmax


def page_bound(q_group: np.ndarray, kmin: np.ndarray, kmax: np.ndarray) -> float:
    """U for one page and group: q_group [G][D]; kmin, kmax [D]."""
    return float(np.maximum(q_group * kmax[None, :], q_group * kmin[None, :]).sum())


def select_pages(c: Cache, kmin, kmax, q: np.ndarray, top_pages: int, b: int, g: int):
    """Selected block indices (ascending) for sequence b, group g; q [Hq][D] fp64."""
    G = q.shape[0] // c.Hkv
    nb = cdiv(int(c.ctx_len[b]), c.page_size)
    cand = np.arange(nb - 1)
    qg = q[g * G:(g + 1) * G]
    U = np.array([page_bound(qg, kmin[c.block_table[b, i], g], kmax[c.block_table[b, i], g])
                  for i in cand])
    chosen = rank(U, cand)[:top_pages]
    return np.sort(np.concatenate([chosen, [nb - 1]])).astype(np.int64), U
