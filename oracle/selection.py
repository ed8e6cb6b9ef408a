"""Selection of the entries to retain (oracle; test infrastructure only).

Per-KV-head top-k (SparseEngine "How it works": SnapKV selection after the
last prompt chunk; H2O's accumulated-score heavy hitters):

    candidates = [cand_lo, cand_hi) minus the forced range
    rank candidates by (pooled score descending, slot ascending)  -- the tie
    rule "lower index first"; keep the first k, plus every slot of the
    forced range [force_lo, force_hi) (observation window / recent tokens /
    protected tail).  Output: kept slots, ascending.

Kara Token2Chunk (KARA Method sections 1-2): top-K discrete candidates of the
compressible window; consecutive candidates (sorted by index) are chunk end
points; chunks are scored from their length and end-point scores and selected
into spans.  The chunk score is fixed by the workload text as
(s_a + s_b)/2 - coef*(b - a).  Readings:

reading (v)    candidates are always retained; a chunk costs its interior,
               b - a - 1 tokens.
reading (vi)   chunks are visited by (chunk score desc, a asc) and added when
               they fit the budget; a misfit is skipped, not a stop.
reading (vii)  if fewer than ``budget`` tokens are retained after the chunks,
               the highest-scoring remaining single tokens (same tie rule) top
               the set up to exactly ``budget``.  (parity unpinned: the pages
               do not say what happens when chunks cannot fill the budget.)

H2O evict-one (SparseEngine "What it is": H2O keeps persistent accumulated
attention scores and evicts physically during generation):

reading (ix)   among resident entries whose position is below the recent
               boundary, evict the lowest accumulated score; ties evict the
               higher position.  Only when the resident count exceeds the
               budget.  (parity unpinned for the tie rule.)
"""
from __future__ import annotations

import numpy as np

from .scoring import avg_pool


def rank(scores: np.ndarray, slots: np.ndarray) -> np.ndarray:
    """Slots ordered by (score descending, slot ascending)."""
    order = np.lexsort((slots, -scores))
    return slots[order]


def topk_keep(s_range: np.ndarray, cand_lo: int, k: int, pool: int,
              force_lo: int, force_hi: int) -> np.ndarray:
    """Kept slots for one (sequence, KV head).

    s_range: scores of slots [cand_lo, cand_lo + len(s_range)).
    """
    pooled = avg_pool(s_range, pool)
    slots = np.arange(cand_lo, cand_lo + len(s_range))
    is_cand = ~((slots >= force_lo) & (slots < force_hi))
    chosen = rank(pooled[is_cand], slots[is_cand])[:k]
    forced = np.arange(force_lo, force_hi)
    return np.sort(np.concatenate([chosen, forced])).astype(np.int64)


def kara_keep(s_range: np.ndarray, cand_lo: int, n_cand: int, budget: int, coef: float,
              force_lo: int, force_hi: int) -> np.ndarray:
    """Token2Chunk retention for one (sequence, KV head): ``budget`` compressible
    slots plus the forced (protected) range, ascending."""
    s_range = np.asarray(s_range, dtype=np.float64)
    n = len(s_range)
    slots = np.arange(cand_lo, cand_lo + n)
    budget = min(budget, n)
    cand = np.sort(rank(s_range, slots)[:n_cand])          # c_1 < ... < c_m
    score = lambda j: s_range[j - cand_lo]                 # noqa: E731
    retained = set(int(c) for c in cand)
    chunks = [(int(a), int(b)) for a, b in zip(cand[:-1], cand[1:])]
    chunk_score = np.array([(score(a) + score(b)) / 2.0 - coef * (b - a) for a, b in chunks])
    order = np.lexsort((np.array([a for a, _ in chunks]), -chunk_score)) if chunks else []
    for i in order:
        a, b = chunks[i]
        interior = b - a - 1
        if interior and len(retained) + interior <= budget:
            retained.update(range(a + 1, b))
    if len(retained) < budget:                              # reading (vii)
        rest = np.array([j for j in slots if j not in retained], dtype=np.int64)
        retained.update(int(j) for j in rank(s_range[rest - cand_lo], rest)[: budget - len(retained)])
    forced = list(range(force_lo, force_hi))
    return np.array(sorted(retained) + forced, dtype=np.int64)


def h2o_victim(acc_row: np.ndarray, pos_row: np.ndarray, ctx: int, budget: int,
               recent_from: int) -> int:
    """Victim slot for one (sequence, KV head), or -1 when ctx <= budget.

    acc_row: accumulated scores of resident slots; pos_row: their positions;
    entries with position >= recent_from are never evicted.
    """
    if ctx <= budget:
        return -1
    slots = np.arange(ctx)
    eligible = pos_row[:ctx] < recent_from
    cand = slots[eligible]
    if len(cand) == 0:
        return -1
    # lowest score first; among equal scores the higher position goes
    order = np.lexsort((-pos_row[cand], acc_row[cand]))
    return int(cand[order[0]])
