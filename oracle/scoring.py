"""Window scoring and pooling (oracle; test infrastructure only).

What is computed (SparseEngine "How it works": SnapKV selects after the last
prompt chunk and H2O evicts with accumulated attention scores; KARA Method
section 1: all window queries score the compressible keys with bidirectional
attention and the weights are accumulated):

    for each sequence b and KV group g (the query heads h with h // G == g):
        A_h = softmax_j( Q_win,h . K_j / sqrt(d) )   over the visible keys j
        s[b, g, j] = sum_{h in g} sum_{q in window} A_h[q, j]

Visibility: causal -- query at logical position t sees the resident keys whose
position (slot map) is <= t; bidirectional -- every query sees every key of
the attention range.

reading (i)    the softmax runs over the whole attention range (for SnapKV
               that includes the window's own visible keys); column sums are
               written only for the output range (the scored prefix).
reading (ii)   Kara: softmax over all window keys, protected tail included;
               only the compressible columns are written.
reading (iii)  scores are sums over heads and queries, not means.
reading (xviii) a query that sees no key of the range contributes nothing.

Pooling (SnapKV workloads): avg_pool1d with an odd kernel k, stride 1, over
the output range only -- reading: zero padding (k-1)/2 on both sides, divisor
always k, output length = input length.
"""
from __future__ import annotations

import numpy as np

from .cache import Cache, values


def _q_values(q_win) -> np.ndarray:
    """q_win: torch tensor or raw-bit / float numpy array [B][w][Hq][D]."""
    if hasattr(q_win, "detach"):
        from .cache import _bits
        return values(_bits(q_win))
    if q_win.dtype in (np.uint16, np.uint32):
        return values(q_win)
    return np.asarray(q_win, dtype=np.float64)


def group_scores(Q: np.ndarray, q_pos: np.ndarray, K: np.ndarray, k_pos: np.ndarray,
                 causal: bool) -> np.ndarray:
    """Column sums of the row softmax for one (sequence, KV group).

    Q: [w][G][D] window queries of the group's heads; q_pos: [w];
    K: [n][D] keys of the attention range; k_pos: [n] their positions.
    Returns s[n] = sum_{q, h} softmax_j(Q[q,h] . K[j] / sqrt(D)).
    """
    w, G, D = Q.shape
    logits = np.einsum("qhd,jd->qhj", Q, K) / np.sqrt(D)           # [w][G][n]
    if causal:
        visible = k_pos[None, :] <= q_pos[:, None]                   # [w][n]
    else:
        visible = np.ones((w, K.shape[0]), dtype=bool)
    visible = np.broadcast_to(visible[:, None, :], logits.shape)
    logits = np.where(visible, logits, -np.inf)
    any_visible = visible.any(axis=2, keepdims=True)
    m = np.where(any_visible, logits.max(axis=2, keepdims=True, initial=-np.inf), 0.0)
    e = np.where(visible, np.exp(logits - m), 0.0)
    denom = e.sum(axis=2, keepdims=True)
    p = np.where(any_visible, e / np.where(denom > 0, denom, 1.0), 0.0)
    return p.sum(axis=(0, 1))


def score_window(c: Cache, q_win, q_pos, attn_lo, attn_hi, out_lo, out_hi,
                 causal: bool, groups=None) -> dict:
    """Scores s[b][g][j] for j in [out_lo[b], out_hi[b]) (resident-slot indices).

    q_win [B][w][Hq][D]; q_pos [B][w] logical positions of the window queries;
    the softmax runs over resident slots [attn_lo[b], attn_hi[b]).  Returns
    {(b, g): array over the output range}.  ``groups`` limits the (b, g) pairs.
    """
    Qv = _q_values(q_win)
    q_pos = np.asarray(q_pos.cpu() if hasattr(q_pos, "cpu") else q_pos, dtype=np.int64)
    B, w, Hq, D = Qv.shape
    G = Hq // c.Hkv
    out = {}
    pairs = groups if groups is not None else [(b, g) for b in range(B) for g in range(c.Hkv)]
    for b, g in pairs:
        lo, hi = int(attn_lo[b]), int(attn_hi[b])
        olo, ohi = int(out_lo[b]), int(out_hi[b])
        assert lo <= olo <= ohi <= hi
        slots = np.arange(lo, hi)
        K = c.keys(b, g, slots)
        k_pos = c.slot_map[b, g, lo:hi]
        s = group_scores(Qv[b, :, g * G:(g + 1) * G, :], q_pos[b], K, k_pos, causal)
        out[(b, g)] = s[olo - lo: ohi - lo]
    return out


def avg_pool(x: np.ndarray, kernel: int) -> np.ndarray:
    """avg_pool1d, stride 1, zero padding (kernel-1)/2 each side, divisor kernel."""
    assert kernel % 2 == 1
    if kernel == 1:
        return x.astype(np.float64).copy()
    pad = kernel // 2
    xp = np.concatenate([np.zeros(pad), np.asarray(x, dtype=np.float64), np.zeros(pad)])
    out = np.zeros(len(x))
    for i in range(len(x)):
        out[i] = xp[i:i + kernel].sum() / kernel
    return out
