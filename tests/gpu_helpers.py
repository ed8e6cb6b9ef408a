"""Drivers for the GPU parity tests: run one stage through the C-ABI binding
and compare with the oracle under the stated parity rules.

Rules (fixed by the method statement):
  * block tables, slot maps, context lengths, free lists and kept index sets
    match bit-exactly; a kept-set difference is allowed only for indices whose
    oracle score is within 1e-6 relative of the oracle's k-th score;
  * scores: 1e-3 relative for bf16 inputs, 1e-5 for fp32; oracle scores below
    1e-12 * w * G are compared absolutely at that floor (reading (xvi));
  * decode outputs: 2e-2 absolute for bf16, 1e-5 for fp32.
"""
from __future__ import annotations

import numpy as np
import torch

import attention_scored_sparse_gb300 as se
from oracle import cache as ocache
from oracle import selection as osel
from oracle import scoring as oscore

SCORE_RTOL = {torch.bfloat16: 1e-3, torch.float32: 1e-5}
OUT_ATOL = {torch.bfloat16: 2e-2, torch.float32: 1e-5}
TIE_REL = 1e-6


def status(cache) -> int:
    return int(cache.status.item())


def keep_tensor(keep, B, H, width, device):
    t = torch.full((B, H, max(width, 1)), -1, dtype=torch.int32)
    for b in range(B):
        for h in range(H):
            k = np.asarray(keep[b][h])
            t[b, h, : len(k)] = torch.from_numpy(k.astype(np.int32))
    return t.to(device)


def random_keep(c: ocache.Cache, seed: int, first=None, frac=None):
    """Generator-side keep lists (input construction only)."""
    rng = np.random.default_rng(seed)
    keep, firsts = [], []
    for b in range(c.B):
        ctx = int(c.ctx_len[b])
        f = int(rng.integers(0, ctx + 1)) if first is None else first[b]
        n = int(rng.integers(0, ctx - f + 1)) if frac is None else int((ctx - f) * frac)
        keep.append([np.sort(rng.choice(np.arange(f, ctx), n, replace=False)) for _ in range(c.Hkv)])
        firsts.append(f)
    return keep, firsts


def assert_cache_equal(pc, c: ocache.Cache, seqs=None, data=True, data_seqs=None):
    """GPU cache tensors == oracle cache, bit for bit.  Slot maps of ``seqs``
    (every sequence by default), K/V bytes of ``data_seqs`` (default: seqs)."""
    np.testing.assert_array_equal(pc.block_table.cpu().numpy(), c.block_table)
    np.testing.assert_array_equal(pc.ctx_len.cpu().numpy(), c.ctx_len)
    np.testing.assert_array_equal(pc.logical_len.cpu().numpy(), c.logical_len)
    top = int(pc.free_top.item())
    assert top == c.free_top
    np.testing.assert_array_equal(pc.free_list[:top].cpu().numpy(), c.free_list[:top])
    np.testing.assert_array_equal(pc.page_refcount.cpu().numpy(), c.page_refcount)
    sm = pc.slot_map.cpu().numpy()
    bs = range(c.B) if seqs is None else seqs
    for b in bs:
        np.testing.assert_array_equal(sm[b], c.slot_map[b])
    if data:
        for b in (bs if data_seqs is None else data_seqs):
            ctx = int(c.ctx_len[b])
            if ctx == 0:
                continue
            slots = np.arange(ctx)
            pages = c.block_table[b, slots // c.page_size]
            rows = slots % c.page_size
            pi = torch.as_tensor(pages, device=pc.k_pool.device)
            ri = torch.as_tensor(rows, device=pc.k_pool.device)
            gk = ocache._bits(pc.k_pool[pi, :, ri, :])
            gv = ocache._bits(pc.v_pool[pi, :, ri, :])
            np.testing.assert_array_equal(gk, c.k[pages, :, rows, :])
            np.testing.assert_array_equal(gv, c.v[pages, :, rows, :])


def assert_scores_close(gpu_row, oracle_row, dtype, w, G):
    floor = 1e-12 * w * G
    g = np.asarray(gpu_row, dtype=np.float64)
    o = np.asarray(oracle_row, dtype=np.float64)
    err = np.abs(g - o) / np.maximum(np.abs(o), floor)
    assert err.max() <= SCORE_RTOL[dtype], (err.max(), int(err.argmax()))


def assert_keep_near(gpu_keep, oracle_keep, ranking_scores: dict, k: int, forced=()):
    """Kept sets equal, or differing only at oracle near-ties of the k-th score.

    ranking_scores: {slot: oracle score used for ranking} over the candidates.
    """
    gs, os_ = set(int(x) for x in gpu_keep), set(int(x) for x in oracle_keep)
    assert list(gpu_keep) == sorted(gs), "GPU keep list not ascending"
    assert len(gs) == len(os_)
    if gs == os_:
        return 0
    assert set(forced) <= gs
    ranked = sorted(ranking_scores.items(), key=lambda kv: (-kv[1], kv[0]))
    kth = ranked[k - 1][1]
    for j in gs ^ os_:
        assert j in ranking_scores, j
        assert abs(ranking_scores[j] - kth) <= TIE_REL * abs(kth), (j, ranking_scores[j], kth)
    return len(gs ^ os_) // 2


def pooled_scores(s_range, cand_lo, pool):
    pooled = oscore.avg_pool(s_range, pool)
    return {cand_lo + i: float(v) for i, v in enumerate(pooled)}


def run_decode(pc, Hq, q, view, sel=None, n_sel=0, acc=None, max_entries=None):
    kv = se.kv_desc(pc, Hq)
    o = torch.empty_like(q)
    if max_entries is None:
        if view == se.SE_VIEW_DENSE:
            max_entries = int(pc.ctx_len.max().item())
        elif view == se.SE_VIEW_PAGES:
            max_entries = n_sel * pc.page_size
        else:
            max_entries = n_sel
    se.se_sparse_decode_attn(kv, q, view=view, o=o, max_entries=max(max_entries, 1), sel=sel,
                             n_sel=n_sel, acc_scores=acc)
    return o


def ranges(B, lo, hi, device="cuda"):
    lo_t = torch.as_tensor(np.broadcast_to(np.asarray(lo), (B,)).astype(np.int32)).to(device)
    hi_t = torch.as_tensor(np.broadcast_to(np.asarray(hi), (B,)).astype(np.int32)).to(device)
    return lo_t, hi_t


def topk_oracle_keep(scores_rows: dict, cand_lo, cand_hi, k, pool, flo, fhi):
    out = {}
    for (b, h), row in scores_rows.items():
        out[(b, h)] = osel.topk_keep(row, cand_lo[b], k, pool, flo[b], fhi[b])
    return out
