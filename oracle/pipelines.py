"""The five workloads end to end, step by step (oracle; test infrastructure).

Each function follows the call order the pages give (SparseEngine "How it
works": finish_step for SnapKV / H2O at the end of prefill, then the decode
selection hooks; KARA Method section 3: periodic compression of the trailing
window) and returns every intermediate so tests can compare stage by stage.
``groups`` / ``seqs`` restrict the float work and the data movement to a
sample of (sequence, KV head) pairs / sequences for full-size checks.
"""
from __future__ import annotations

import numpy as np

from . import attention, cache, quest, scoring, selection
from .cache import Cache, values


def to_f64(t) -> np.ndarray:
    """Torch tensor (bf16 / fp32) or numpy array -> fp64 values."""
    if hasattr(t, "detach"):
        return values(cache._bits(t))
    return np.asarray(t, dtype=np.float64)


def snapkv_select(c: Cache, q_win, q_pos, shape):
    """SnapKV after the last prompt chunk, first half: window scores of the
    scored prefix and the pooled top-k plus the window, per KV head."""
    B, ctx, w = c.B, int(c.ctx_len[0]), shape.window
    scored = ctx - w
    s = scoring.score_window(c, q_win, q_pos, [0] * B, [ctx] * B, [0] * B, [scored] * B,
                             causal=True)
    keep = [[selection.topk_keep(s[(b, h)], 0, shape.keep_topk, shape.pool_kernel, scored, ctx)
             for h in range(c.Hkv)] for b in range(B)]
    return dict(scores=s, keep=keep)


def snapkv_finish(c: Cache, keep, q_dec, groups=None):
    """Second half: compaction of the kept entries from slot 0, then decode
    attention of one query per head over the compacted cache."""
    st = cache.compact(c, keep, [0] * c.B)
    assert st == cache.SE_OK
    o, _ = attention.decode_attention(c, to_f64(q_dec), "dense", groups=groups)
    return o


def snapkv(c: Cache, q_win, q_pos, q_dec, shape):
    """SnapKV after the last prompt chunk: score, pool + top-k, compact, decode."""
    r = snapkv_select(c, q_win, q_pos, shape)
    r["o"] = snapkv_finish(c, r["keep"], q_dec)
    return r


def quest_select(c: Cache, kmin, kmax, q, top_pages: int, groups=None):
    """Quest page selection of one decode step: page bounds, top pages plus
    the current page, per (sequence, KV group)."""
    qv = to_f64(q)
    pairs = groups if groups is not None else [(b, g) for b in range(c.B) for g in range(c.Hkv)]
    sel = {}
    bounds = {}
    for b, g in pairs:
        sel[(b, g)], bounds[(b, g)] = quest.select_pages(c, kmin, kmax, qv[b], top_pages, b, g)
    return dict(sel=sel, bounds=bounds)


def quest_attend(c: Cache, q, sel: dict):
    """Decode attention of one Quest step over the pages ``sel[(b, g)]``."""
    pairs = list(sel)
    selb = {b: {g: sel[(b, g)] for (bb, g) in sel if bb == b} for b in {p[0] for p in pairs}}
    o, _ = attention.decode_attention(c, to_f64(q), "pages", selb, groups=pairs)
    return o


def quest_step(c: Cache, kmin, kmax, q, top_pages: int, groups=None):
    """One Quest decode step: page bound, top pages + current page, attention."""
    r = quest_select(c, kmin, kmax, q, top_pages, groups)
    r["o"] = quest_attend(c, q, r["sel"])
    return r


def h2o_prefill_select(c: Cache, q_prompt, q_pos, shape, acc: np.ndarray, groups=None):
    """H2O at the end of prefill, reading (viii), first half: causal scores
    of the whole prompt become the initial running scores; keep the top
    ``heavy`` of the non-recent prefix plus the ``recent`` last tokens."""
    B, ctx = c.B, int(c.ctx_len[0])
    s = scoring.score_window(c, q_prompt, q_pos, [0] * B, [ctx] * B, [0] * B, [ctx] * B,
                             causal=True, groups=groups)
    for (b, h), v in s.items():
        acc[b, h, :ctx] = v
    keep = [[None] * c.Hkv for _ in range(B)]
    for (b, h), v in s.items():
        keep[b][h] = selection.topk_keep(v[: ctx - shape.recent], 0, shape.heavy, 1,
                                         ctx - shape.recent, ctx)
    return dict(scores=s, keep=keep)


def h2o_prefill(c: Cache, q_prompt, q_pos, shape, acc: np.ndarray):
    """H2O at the end of prefill: scores, selection, compaction from slot 0
    (the running scores move with their entries)."""
    r = h2o_prefill_select(c, q_prompt, q_pos, shape, acc)
    st = cache.compact(c, r["keep"], [0] * c.B, aux=acc)
    assert st == cache.SE_OK
    return r


def h2o_prefill_chunk(c: Cache, acc: np.ndarray, q_chunk, q_pos, k_chunk, v_chunk,
                      heavy: int, recent: int):
    """One chunk of H2O chunk-wise prefill eviction (SparseEngine "How it
    works": H2O evicts during prefill, chunk by chunk, on accumulated scores).

    Reading (xix): the chunk's keys and values are written first; its
    queries then attend causally to every resident entry (earlier survivors
    and the chunk itself) and their group-summed weights are added to the
    running scores (new entries start at 0); when more than heavy + recent
    entries are resident, the top ``heavy`` of the non-recent ones by
    running score (lower slot first on ties) and the last ``recent`` are
    kept and compacted from slot 0, the scores moving with their entries.
    """
    st = cache.append_tokens(c, cache._bits(k_chunk), cache._bits(v_chunk), aux=acc)
    assert st == cache.SE_OK
    B, ctx = c.B, int(c.ctx_len[0])
    s = scoring.score_window(c, q_chunk, q_pos, [0] * B, [ctx] * B, [0] * B, [ctx] * B,
                             causal=True)
    for (b, h), v in s.items():
        acc[b, h, :ctx] += v
    acc_pre = acc.copy()
    keep = None
    if ctx > heavy + recent:
        keep = [[selection.topk_keep(acc[b, h, : ctx - recent], 0, heavy, 1, ctx - recent, ctx)
                 for h in range(c.Hkv)] for b in range(B)]
        st = cache.compact(c, keep, [0] * B, aux=acc)
        assert st == cache.SE_OK
    return dict(acc_pre=acc_pre, keep=keep)


def h2o_step_attend(c: Cache, acc: np.ndarray, q, k_new, v_new, groups=None):
    """First half of an H2O decode step: append this step's key and value,
    dense attention over the resident entries, and this step's group-summed
    weights added to the running scores (the new entry starts at its own
    weight).  ``groups`` limits the float work to those (sequence, KV head)
    pairs; the append is done for every sequence."""
    kb, vb = cache._bits(k_new), cache._bits(v_new)
    st = cache.append(c, kb, vb, aux=acc)
    assert st == cache.SE_OK
    o, psums = attention.decode_attention(c, to_f64(q), "dense", groups=groups)
    for (b, g), (slots, p) in psums.items():
        acc[b, g, slots] += p
    return o


def h2o_victims(c: Cache, acc: np.ndarray, shape, seqs=None) -> np.ndarray:
    """Evict-one choice per (sequence, KV head) after the scores are added
    (-1: within budget); sequences outside ``seqs`` get -1."""
    victim = np.full((c.B, c.Hkv), -1, dtype=np.int64)
    for b in (range(c.B) if seqs is None else seqs):
        recent_from = int(c.logical_len[b]) - shape.recent
        for g in range(c.Hkv):
            victim[b, g] = selection.h2o_victim(acc[b, g], c.slot_map[b, g], int(c.ctx_len[b]),
                                                shape.budget, recent_from)
    return victim


def h2o_step(c: Cache, acc: np.ndarray, q, k_new, v_new, shape):
    """One H2O decode step: append, dense attention, add this step's
    group-summed weights to the running scores, evict one if over budget."""
    o = h2o_step_attend(c, acc, q, k_new, v_new)
    acc_pre = acc.copy()
    victim = h2o_victims(c, acc, shape)
    st = cache.move_last(c, victim, aux=acc)
    assert st == cache.SE_OK
    return dict(o=o, victim=victim, acc_pre=acc_pre)


def kara_compress(c: Cache, q_win, q_pos, shape, groups=None, seqs=None):
    """Kara periodic compression of the trailing window: bidirectional scores of
    the compressible keys, Token2Chunk retention, compaction from the window."""
    B = c.B
    ctx = [int(x) for x in c.ctx_len]
    win_lo = [x - shape.window for x in ctx]
    prot_lo = [x - shape.protected for x in ctx]
    s = scoring.score_window(c, q_win, q_pos, win_lo, ctx, win_lo, prot_lo, causal=False,
                             groups=groups)
    keep = [[None] * c.Hkv for _ in range(B)]
    for b in range(B):
        for h in range(c.Hkv):
            if (b, h) in s:
                keep[b][h] = selection.kara_keep(s[(b, h)], win_lo[b], shape.candidates,
                                                 shape.budget, shape.chunk_coef, prot_lo[b], ctx[b])
    return dict(scores=s, keep=keep, first_slot=win_lo)


def kara_schedule_step(c: Cache, q, k_new, v_new, q_ring, win_start, shape):
    """One step of Kara compression inside a decode loop (KARA Method,
    periodic compression of the trailing window; reading (xxvi): the window
    compresses when the appended token fills it, after that step's attention;
    its queries are those of its own positions, which the caller keeps in
    q_ring at slot position % window).  Sequences whose window is not full
    are left as they are.  win_start (list) is updated in place."""
    B, W = c.B, shape.window
    for b in range(B):
        q_ring[b, int(c.logical_len[b]) % W] = q[b]
    st = cache.append(c, cache._bits(k_new), cache._bits(v_new))
    assert st == cache.SE_OK
    o, _ = attention.decode_attention(c, to_f64(q), "dense")
    ctx = [int(x) for x in c.ctx_len]
    due = [b for b in range(B) if ctx[b] - win_start[b] >= W]
    keep_all, scores = None, {}
    if due:
        win_lo = [ctx[b] - W if b in due else ctx[b] for b in range(B)]
        prot_lo = [ctx[b] - shape.protected if b in due else ctx[b] for b in range(B)]
        q_pos = np.array([[int(c.logical_len[b]) - W + i for i in range(W)] for b in range(B)])
        groups = [(b, h) for b in due for h in range(c.Hkv)]
        scores = scoring.score_window(c, q_ring, q_pos, win_lo, ctx, win_lo, prot_lo,
                                      causal=False, groups=groups)
        keep_all = [[np.array([], dtype=np.int64)] * c.Hkv for _ in range(B)]
        for b in due:
            keep_all[b] = [selection.kara_keep(scores[(b, h)], win_lo[b], shape.candidates,
                                               shape.budget, shape.chunk_coef, prot_lo[b], ctx[b])
                           for h in range(c.Hkv)]
        st = cache.compact(c, keep_all, win_lo)
        assert st == cache.SE_OK
    return dict(o=o, due=due, keep=keep_all, scores=scores)
