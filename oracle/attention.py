"""Decode attention over a view of the cache (oracle; test infrastructure only).

SparseEngine "How it works" (AttentionView): View = BuildView(C, I),
o = Attention(q, View).  For each query head h of KV group g:

    o_h = sum_j softmax_j(q_h . k_j / sqrt(d)) v_j      over the view's entries

Views: every resident entry (dense), the resident slots of a list of blocks
(pages), or a list of resident slots (tokens).  Alongside o this returns, per
(b, g), the group-summed probabilities sum_{h in g} p_{h,j} of every entry --
what an H2O step adds to its running scores.
"""
from __future__ import annotations

import numpy as np

from .cache import Cache


def view_slots(c: Cache, b: int, g: int, view: str, sel=None) -> np.ndarray:
    ctx = int(c.ctx_len[b])
    if view == "dense":
        return np.arange(ctx)
    if view == "pages":
        blocks = np.asarray(sel[b][g])
        blocks = blocks[blocks >= 0]
        P = c.page_size
        s = (blocks[:, None] * P + np.arange(P)[None, :]).reshape(-1)
        return s[s < ctx]
    if view == "tokens":
        s = np.asarray(sel[b][g])
        return s[s >= 0]
    raise ValueError(view)


def attend(q_group: np.ndarray, K: np.ndarray, V: np.ndarray):
    """q_group [G][D], K/V [n][D] -> (o [G][D], p [G][n])."""
    D = q_group.shape[1]
    logits = q_group @ K.T / np.sqrt(D)
    m = logits.max(axis=1, keepdims=True)
    e = np.exp(logits - m)
    p = e / e.sum(axis=1, keepdims=True)
    return p @ V, p


def decode_attention(c: Cache, q: np.ndarray, view: str = "dense", sel=None, groups=None):
    """q [B][Hq][D] fp64 -> (o {(b,g): [G][D]}, psum {(b,g): (slots, sum_h p)})."""
    B, Hq, D = q.shape
    G = Hq // c.Hkv
    outs, psums = {}, {}
    pairs = groups if groups is not None else [(b, g) for b in range(B) for g in range(c.Hkv)]
    for b, g in pairs:
        slots = view_slots(c, b, g, view, sel)
        o, p = attend(q[b, g * G:(g + 1) * G], c.keys(b, g, slots), c.vals(b, g, slots))
        outs[(b, g)] = o
        psums[(b, g)] = (slots, p.sum(axis=0))
    return outs, psums
