"""GPU vs oracle: top-k selection (pooled, forced ranges), Kara Token2Chunk,
H2O evict-one, Quest metadata and page selection, decode attention over the
three views (with H2O score accumulation) and window scoring (causal and
bidirectional, bf16 and fp32).  Sizes span several tiles and ragged tails."""
import json
import os

import numpy as np
import pytest
import torch

import se_workloads as W
from oracle import attention as oattn
from oracle import cache as ocache
from oracle import quest as oquest
from oracle import scoring as oscore
from oracle import selection as osel
from tests import gpu_helpers as H

pytestmark = pytest.mark.gpu
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _desc_dims(se, B, Hkv, dtype=torch.float32):
    """A minimal cache for calls that only need the shape of the descriptor."""
    shape = W.Shape(name="dims", B=B, Hq=Hkv, Hkv=Hkv, D=128, page_size=16, ctx=16, dtype=dtype)
    pc = W.build_paged_cache(shape, num_pages=B + 1, max_ctx=16, device="cuda", tag="dims")
    return pc, se.kv_desc(pc, Hkv)


# ---------------------------------------------------------------------------
# selection
# ---------------------------------------------------------------------------


@pytest.mark.parametrize("n,k,pool,flo,fhi", [
    (480, 96, 7, 480, 512),        # tiny SnapKV shape: window after the candidates
    (5000, 700, 7, 5000, 5064),    # several 1024-element rows, ragged
    (3968, 1024, 1, 3968, 4096),   # H2O prompt shape, no pooling
    (2000, 50, 1, 100, 140),       # forced range inside the candidates
    (300, 400, 3, 300, 301),       # k larger than the candidates
])
def test_topk_matches_oracle(cuda_lib, n, k, pool, flo, fhi):
    se = cuda_lib
    B, Hkv = 3, 2
    pc, kv = _desc_dims(se, B, Hkv)
    g = W.generator("cpu", "topk", n, k)
    scores = torch.rand((B, Hkv, max(n, fhi) + 8), generator=g)
    scores[0, 0, : n // 2] = torch.round(scores[0, 0, : n // 2] * 8) / 8   # exact ties
    sc = scores.cuda()
    keep = torch.full((B, Hkv, k + (fhi - flo) + 4), -7, dtype=torch.int32, device="cuda")
    n_keep = torch.zeros(B, dtype=torch.int32, device="cuda")
    lo, hi = H.ranges(B, 0, n)
    f0, f1 = H.ranges(B, flo, fhi)
    se.se_topk_select(kv, sc, mode=se.SE_SELECT_TOPK, cand_lo=lo, cand_hi=hi, force_lo=f0,
                      force_hi=f1, keep_idx=keep, n_keep=n_keep, pool_kernel=pool, k=k, n_max=n)
    torch.cuda.synchronize()
    assert H.status(pc) == 0
    kg = keep.cpu().numpy()
    ncand = n - max(0, min(fhi, n) - max(flo, 0))
    total = min(k, ncand) + (fhi - flo)
    assert (n_keep.cpu().numpy() == total).all()
    for b in range(B):
        for h in range(Hkv):
            row = scores[b, h, :n].double().numpy()
            ok = osel.topk_keep(row, 0, k, pool, flo, fhi)
            pooled = H.pooled_scores(row, 0, pool)
            cand = {j: v for j, v in pooled.items() if not flo <= j < fhi}
            H.assert_keep_near(kg[b, h, :total], ok, cand, min(k, ncand), range(flo, fhi))
            assert (kg[b, h, total:] == -1).all()


def test_kara_golden_hand_example_on_gpu(cuda_lib):
    se = cuda_lib
    g = json.load(open(os.path.join(GOLDEN, "kara_token2chunk_hand.json")))
    pc, kv = _desc_dims(se, 1, 1)
    scores = torch.zeros((1, 1, 128))
    scores[0, 0, 100:116] = torch.tensor(g["scores"])
    keep = torch.zeros((1, 1, 14), dtype=torch.int32, device="cuda")
    lo, hi = H.ranges(1, 100, 116)
    f0, f1 = H.ranges(1, 116, 120)
    se.se_topk_select(kv, scores.cuda(), mode=se.SE_SELECT_KARA_CHUNK, cand_lo=lo, cand_hi=hi,
                      force_lo=f0, force_hi=f1, keep_idx=keep, k=g["n_cand"],
                      chunk_budget=g["budget"], chunk_coef=g["coef"], n_max=16)
    torch.cuda.synchronize()
    assert keep[0, 0].cpu().tolist() == g["expected"]


@pytest.mark.parametrize("seed", range(3))
def test_kara_matches_oracle(cuda_lib, seed):
    se = cuda_lib
    B, Hkv = 6, 4
    pc, kv = _desc_dims(se, B, Hkv)
    base = 1000
    scores = torch.rand((B, Hkv, base + 256), generator=W.generator("cpu", "kara", seed))
    scores = scores * torch.rand((B, Hkv, 1), generator=W.generator("cpu", "kara_s", seed)) * 50
    keep = torch.zeros((B, Hkv, 96), dtype=torch.int32, device="cuda")
    n_keep = torch.zeros(B, dtype=torch.int32, device="cuda")
    lo, hi = H.ranges(B, base, base + 224)
    f0, f1 = H.ranges(B, base + 224, base + 256)
    se.se_topk_select(kv, scores.cuda(), mode=se.SE_SELECT_KARA_CHUNK, cand_lo=lo, cand_hi=hi,
                      force_lo=f0, force_hi=f1, keep_idx=keep, n_keep=n_keep, k=32,
                      chunk_budget=64, chunk_coef=0.01, n_max=224)
    torch.cuda.synchronize()
    assert (n_keep.cpu().numpy() == 96).all()
    kg = keep.cpu().numpy()
    for b in range(B):
        for h in range(Hkv):
            row = scores[b, h, base:base + 224].double().numpy()
            ok = osel.kara_keep(row, base, 32, 64, 0.01, base + 224, base + 256)
            assert list(kg[b, h]) == list(ok)


def test_evict_one_matches_oracle(cuda_lib):
    se = cuda_lib
    shape = W.Shape(name="ev", B=5, Hq=8, Hkv=4, D=128, page_size=16, ctx=300, dtype=torch.bfloat16)
    pc = W.build_paged_cache(shape, num_pages=100, max_ctx=320, device="cuda", tag="ev")
    pc.logical_len.copy_(torch.tensor([400, 350, 300, 301, 500], dtype=torch.int32))
    pc.ctx_len.copy_(torch.tensor([300, 290, 100, 300, 299], dtype=torch.int32))
    perm = torch.stack([torch.randperm(320, generator=W.generator("cpu", "evp", i)) for i in range(20)])
    pc.slot_map.copy_(perm.view(5, 4, 320).to(torch.int32))
    acc = torch.round(torch.rand((5, 4, 320), generator=W.generator("cpu", "eva")) * 50) / 50
    victim = torch.zeros((5, 4), dtype=torch.int32, device="cuda")
    se.se_topk_select(se.kv_desc(pc, 8), acc.cuda(), mode=se.SE_SELECT_EVICT_ONE,
                      keep_idx=victim, budget=200, recent=64)
    torch.cuda.synchronize()
    c = ocache.from_tensors(pc)
    for b in range(5):
        for h in range(4):
            v = osel.h2o_victim(acc[b, h].double().numpy(), c.slot_map[b, h], int(c.ctx_len[b]),
                                200, int(c.logical_len[b]) - 64)
            assert int(victim[b, h]) == v


# ---------------------------------------------------------------------------
# Quest
# ---------------------------------------------------------------------------


@pytest.mark.parametrize("ctx,top", [(16 * 300 + 7, 40), (16 * 64, 100)])
def test_quest_meta_and_selection_match_oracle(cuda_lib, ctx, top):
    se = cuda_lib
    shape = W.quest_decode(B=2, ctx=ctx, top_pages=top, steps=2)
    inp = W.quest_inputs(shape, "cuda")
    pc = inp["cache"]
    kv = se.kv_desc(pc, shape.Hq)
    kmin = torch.empty_like(pc.k_pool[:, :, 0, :])
    kmax = torch.empty_like(kmin)
    se.se_quest_build_meta(kv, kmin, kmax)
    c = ocache.from_tensors(pc)
    omin, omax = oquest.build_meta(c)
    torch.cuda.synchronize()
    nb = W.cdiv(ctx, 16)
    for b in range(2):
        pages = c.block_table[b, :nb]
        np.testing.assert_array_equal(kmin[pages].double().cpu().numpy(), omin[pages])
        np.testing.assert_array_equal(kmax[pages].double().cpu().numpy(), omax[pages])
    for step in range(2):
        q = inp["q_steps"][step]
        page_idx = torch.full((2, 8, top + 1), -9, dtype=torch.int32, device="cuda")
        n_sel = torch.zeros(2, dtype=torch.int32, device="cuda")
        se.se_quest_page_select(kv, kmin, kmax, q, top_pages=top, max_blocks=nb,
                                page_idx=page_idx, n_sel=n_sel)
        torch.cuda.synchronize()
        qv = q.double().cpu().numpy()
        got = page_idx.cpu().numpy()
        nsel = min(top, nb - 1) + 1
        assert (n_sel.cpu().numpy() == nsel).all()
        for b in range(2):
            for g in range(8):
                sel, U = oquest.select_pages(c, omin, omax, qv[b], top, b, g)
                ranking = {i: float(U[i]) for i in range(nb - 1)}
                H.assert_keep_near(got[b, g, :nsel], sel, ranking, min(top, nb - 1), [nb - 1])
                assert (got[b, g, nsel:] == -1).all()


@pytest.mark.parametrize("Hkv,G,dtype", [(1, 8, torch.bfloat16), (2, 4, torch.bfloat16),
                                         (4, 2, torch.bfloat16), (8, 1, torch.bfloat16),
                                         (2, 4, torch.float32)])
def test_quest_selection_head_layouts_match_oracle(cuda_lib, Hkv, G, dtype):
    """The page bound for every layout of KV heads over a CTA (1, 2, 4 or 8
    heads of a page read together), group sizes 1 to 8, and the fp32 form;
    contexts that end inside a page and span several CTA ranges."""
    se = cuda_lib
    ctx, top = 16 * 1500 + 9, 60
    shape = W.quest_decode(B=2, ctx=ctx, top_pages=top, steps=1, Hq=Hkv * G, Hkv=Hkv, dtype=dtype)
    inp = W.quest_inputs(shape, "cuda")
    pc = inp["cache"]
    pc.ctx_len.copy_(torch.tensor([ctx, ctx - 5000], dtype=torch.int32))
    kv = se.kv_desc(pc, shape.Hq)
    kmin = torch.empty_like(pc.k_pool[:, :, 0, :])
    kmax = torch.empty_like(kmin)
    se.se_quest_build_meta(kv, kmin, kmax)
    c = ocache.from_tensors(pc)
    omin, omax = oquest.build_meta(c)
    nb_max = W.cdiv(ctx, 16)
    q = inp["q_steps"][0]
    page_idx = torch.full((2, Hkv, top + 1), -9, dtype=torch.int32, device="cuda")
    n_sel = torch.zeros(2, dtype=torch.int32, device="cuda")
    se.se_quest_page_select(kv, kmin, kmax, q, top_pages=top, max_blocks=nb_max,
                            page_idx=page_idx, n_sel=n_sel)
    torch.cuda.synchronize()
    assert H.status(pc) == 0
    qv = q.double().cpu().numpy()
    got = page_idx.cpu().numpy()
    for b in range(2):
        nb = W.cdiv(int(c.ctx_len[b]), 16)
        nsel = min(top, nb - 1) + 1
        assert int(n_sel[b].item()) == nsel
        for g in range(Hkv):
            sel, U = oquest.select_pages(c, omin, omax, qv[b], top, b, g)
            ranking = {i: float(U[i]) for i in range(nb - 1)}
            H.assert_keep_near(got[b, g, :nsel], sel, ranking, min(top, nb - 1), [nb - 1])
            assert (got[b, g, nsel:] == -1).all()


# ---------------------------------------------------------------------------
# decode attention
# ---------------------------------------------------------------------------


@pytest.mark.parametrize("dtype,D,G", [(torch.bfloat16, 128, 4), (torch.float32, 64, 4),
                                       (torch.bfloat16, 64, 2), (torch.float32, 128, 8)])
def test_decode_attention_views_match_oracle(cuda_lib, dtype, D, G):
    se = cuda_lib
    B, Hkv = 3, 2
    shape = W.Shape(name="dec", B=B, Hq=Hkv * G, Hkv=Hkv, D=D, page_size=16, ctx=1500, dtype=dtype)
    pc = W.build_paged_cache(shape, num_pages=B * 94 + 3, max_ctx=1500, device="cuda", tag="dec")
    pc.ctx_len.copy_(torch.tensor([1500, 1333, 17], dtype=torch.int32))
    c = ocache.from_tensors(pc)
    q = W.normal((B, shape.Hq, D), dtype, "cuda", "dec", "q", D, G)
    qv = q.double().cpu().numpy()
    rng = np.random.default_rng(D + G)
    sel_p = np.full((B, Hkv, 40), -1, dtype=np.int32)
    sel_t = np.full((B, Hkv, 700), -1, dtype=np.int32)
    for b in range(B):
        nb = W.cdiv(int(c.ctx_len[b]), 16)
        for g in range(Hkv):
            p = np.sort(rng.choice(nb, min(nb, 37), replace=False))
            sel_p[b, g, : len(p)] = p
            t = np.sort(rng.choice(int(c.ctx_len[b]), min(int(c.ctx_len[b]), 650), replace=False))
            sel_t[b, g, : len(t)] = t
    for view, sel, n_sel, oview, osel_ in [
            (se.SE_VIEW_DENSE, None, 0, "dense", None),
            (se.SE_VIEW_PAGES, sel_p, 40, "pages", sel_p),
            (se.SE_VIEW_TOKENS, sel_t, 700, "tokens", sel_t)]:
        acc = torch.zeros((B, Hkv, 1504), device="cuda")
        st = None if sel is None else torch.from_numpy(sel).cuda()
        o = H.run_decode(pc, shape.Hq, q, view, st, n_sel, acc=acc)
        torch.cuda.synchronize()
        oo, ps = oattn.decode_attention(c, qv, oview, osel_)
        og = o.double().cpu().numpy()
        accg = acc.cpu().double().numpy()
        for b in range(B):
            for g in range(Hkv):
                ref = oo[(b, g)]
                err = np.abs(og[b, g * G:(g + 1) * G] - ref).max()
                assert err <= H.OUT_ATOL[dtype], (oview, b, g, err)
                slots, p = ps[(b, g)]
                expect = np.zeros(1504)
                expect[slots] += p
                np.testing.assert_allclose(accg[b, g], expect, rtol=1e-4, atol=1e-6)


def _aligned_ctas(units, max_entries):
    """CTAs of the unit-aligned split of decode attention (chunks of at most
    1024 entries, halved down to 128 while fewer than 152 x 4 CTAs)."""
    chunk = 1024
    while chunk > 128 and units * W.cdiv(max_entries, chunk) < 608:
        chunk //= 2
    return units * W.cdiv(max_entries, chunk)


def _decode_split(units, max_entries, G):
    """The work split decode attention takes for a shape: a cluster of k CTAs
    per (sequence, KV head) unit (k a power of two up to 16, each CTA at most
    1024 entries, the most k that keep the grid within 152 x 4 CTAs), else
    split-K with a merge through global memory, unit-aligned or cut evenly
    ("stream")."""
    se_ = 128 // G
    sp = W.cdiv(max_entries, se_)
    k_cl = 0
    for kc in (1, 2, 4, 8, 16):
        if W.cdiv(sp, kc) > 1024 // se_:
            continue
        if units * kc > 608:
            break
        k_cl = kc
    if k_cl:
        return ("cluster", k_cl)
    n_al = _aligned_ctas(units, max_entries)
    return ("aligned" if n_al <= 608 or n_al >= 4 * 608 else "stream", n_al)


@pytest.mark.parametrize("B,Hkv,G,D,me,path", [
    (40, 8, 4, 64, 600, ("cluster", 1)),
    (20, 8, 4, 128, 1153, ("cluster", 2)),
    (10, 8, 4, 64, 3000, ("cluster", 4)),
    (5, 8, 4, 64, 5000, ("cluster", 8)),
    (2, 2, 4, 128, 9000, ("cluster", 16)),
    (4, 4, 8, 128, 5000, ("cluster", 16)),
    (40, 8, 4, 128, 1153, ("stream", 640)),
    (2, 2, 4, 128, 20000, ("stream", 628)),
    (1, 2, 4, 128, 20000, ("aligned", 314)),
])
def test_decode_attention_splits_match_oracle(cuda_lib, B, Hkv, G, D, me, path):
    """Every work split of decode attention against the oracle: clusters of
    1 to 16 CTAs per unit merging through shared memory, and for grids of
    more than one wave or views longer than 16 x 1024 entries split-K with
    the merge in global memory (ranges aligned to units, or cut evenly across
    unit boundaries).  Ragged contexts (one of a single token, one of 16),
    dense view with running scores and a token view."""
    se = cuda_lib
    assert _decode_split(B * Hkv, me, G) == path
    dtype = torch.bfloat16
    tag = f"dsplit{B}_{me}"
    shape = W.Shape(name=tag, B=B, Hq=Hkv * G, Hkv=Hkv, D=D, page_size=16, ctx=me, dtype=dtype)
    pc = W.build_paged_cache(shape, num_pages=B * W.cdiv(me, 16) + 3, max_ctx=me, device="cuda",
                             tag=tag)
    rng = np.random.default_rng(me + B)
    ctx = rng.integers(1, me + 1, size=B).astype(np.int32)
    ctx[:3] = [me, 1, 16][:B]
    pc.ctx_len.copy_(torch.from_numpy(ctx))
    c = ocache.from_tensors(pc)
    q = W.normal((B, shape.Hq, D), dtype, "cuda", tag, "q")
    qv = q.double().cpu().numpy()
    n_tok = 1100
    sel_t = np.full((B, Hkv, n_tok), -1, dtype=np.int32)
    for b in range(B):
        for g in range(Hkv):
            t = np.sort(rng.choice(int(ctx[b]), min(int(ctx[b]), 1000), replace=False))
            sel_t[b, g, : len(t)] = t
    stride = W.cdiv(me, 16) * 16
    for view, sel, n_sel, oview in [(se.SE_VIEW_DENSE, None, 0, "dense"),
                                    (se.SE_VIEW_TOKENS, sel_t, n_tok, "tokens")]:
        acc = torch.zeros((B, Hkv, stride), device="cuda")
        st = None if sel is None else torch.from_numpy(sel).cuda()
        o = H.run_decode(pc, shape.Hq, q, view, st, n_sel, acc=acc)
        torch.cuda.synchronize()
        assert int(pc.status.item()) == 0
        oo, ps = oattn.decode_attention(c, qv, oview, sel)
        og = o.double().cpu().numpy()
        accg = acc.cpu().double().numpy()
        for b in range(B):
            for g in range(Hkv):
                err = np.abs(og[b, g * G:(g + 1) * G] - oo[(b, g)]).max()
                assert err <= H.OUT_ATOL[dtype], (oview, b, g, err)
                slots, p = ps[(b, g)]
                expect = np.zeros(stride)
                expect[slots] += p
                np.testing.assert_allclose(accg[b, g], expect, rtol=1e-4, atol=1e-6)


def test_decode_attention_repeats_bit_for_bit(cuda_lib):
    """The cluster merge sums the partials of an element in a fixed order and
    the split-K merge in the order of the partial slots: repeated calls give
    the same output and running scores bit for bit."""
    se = cuda_lib
    for B, Hkv, me in [(2, 2, 9000), (2, 2, 20000)]:
        tag = f"drep{me}"
        shape = W.Shape(name=tag, B=B, Hq=Hkv * 4, Hkv=Hkv, D=128, page_size=16, ctx=me,
                        dtype=torch.bfloat16)
        pc = W.build_paged_cache(shape, num_pages=B * W.cdiv(me, 16) + 3, max_ctx=me,
                                 device="cuda", tag=tag)
        q = W.normal((B, shape.Hq, 128), torch.bfloat16, "cuda", tag, "q")
        outs = []
        for _ in range(3):
            acc = torch.zeros((B, Hkv, me), device="cuda")
            outs.append((H.run_decode(pc, shape.Hq, q, se.SE_VIEW_DENSE, acc=acc), acc))
        torch.cuda.synchronize()
        assert int(pc.status.item()) == 0
        for o, acc in outs[1:]:
            assert torch.equal(o, outs[0][0]) and torch.equal(acc, outs[0][1])


def test_decode_attention_special_cases(cuda_lib):
    se = cuda_lib
    shape = W.Shape(name="dsc", B=2, Hq=4, Hkv=1, D=128, page_size=16, ctx=40, dtype=torch.float32)
    pc = W.build_paged_cache(shape, num_pages=8, max_ctx=40, device="cuda", tag="dsc")
    q = W.normal((2, 4, 128), torch.float32, "cuda", "dsc", "q")
    # one token: output is that token's value
    sel = torch.tensor([[[7]], [[33]]], dtype=torch.int32, device="cuda")
    o = H.run_decode(pc, 4, q, se.SE_VIEW_TOKENS, sel, 1)
    c = ocache.from_tensors(pc)
    torch.cuda.synchronize()
    for b, s in [(0, 7), (1, 33)]:
        np.testing.assert_allclose(o[b].cpu().numpy(), np.repeat(c.vals(b, 0, [s]), 4, 0), rtol=1e-6)
    # constant V: output is the constant
    pc.v_pool.fill_(0.625)
    o = H.run_decode(pc, 4, q, se.SE_VIEW_DENSE)
    torch.cuda.synchronize()
    np.testing.assert_allclose(o.cpu().numpy(), 0.625, rtol=1e-6)


# ---------------------------------------------------------------------------
# window scoring
# ---------------------------------------------------------------------------


@pytest.mark.parametrize("dtype,D,G,causal", [
    (torch.float32, 64, 4, True), (torch.bfloat16, 128, 4, True),
    (torch.bfloat16, 128, 4, False), (torch.float32, 128, 2, False), (torch.bfloat16, 64, 8, True)])
def test_score_window_matches_oracle(cuda_lib, dtype, D, G, causal):
    se = cuda_lib
    B, Hkv, w = 2, 2, 45
    ctx = 700
    shape = W.Shape(name="sc", B=B, Hq=Hkv * G, Hkv=Hkv, D=D, page_size=16, ctx=ctx, dtype=dtype)
    pc = W.build_paged_cache(shape, num_pages=B * 44 + 2, max_ctx=ctx, device="cuda", tag="sc")
    q_win = W.normal((B, w, shape.Hq, D), dtype, "cuda", "sc", "q", D, G)
    q_pos = torch.arange(ctx - w, ctx, dtype=torch.int32).repeat(B, 1)
    q_pos[1] -= 100                          # a window inside the context for sequence 1
    q_pos = q_pos.cuda()
    attn_lo, attn_hi = [3, 0], [ctx, ctx - 37]
    out_lo, out_hi = [10, 0], [ctx - w, ctx - 37]
    scores = torch.full((B, Hkv, ctx + 4), -5.0, device="cuda")
    se.se_score_window(se.kv_desc(pc, shape.Hq), q_win, q_pos,
                       torch.tensor(attn_lo, dtype=torch.int32, device="cuda"),
                       torch.tensor(attn_hi, dtype=torch.int32, device="cuda"),
                       torch.tensor(out_lo, dtype=torch.int32, device="cuda"),
                       torch.tensor(out_hi, dtype=torch.int32, device="cuda"),
                       causal=causal, accumulate=False, n_max=ctx, scores=scores)
    torch.cuda.synchronize()
    c = ocache.from_tensors(pc)
    os_ = oscore.score_window(c, q_win, q_pos.cpu().numpy(), attn_lo, attn_hi, out_lo, out_hi, causal)
    sg = scores.cpu().double().numpy()
    for (b, g), row in os_.items():
        H.assert_scores_close(sg[b, g, out_lo[b]:out_hi[b]], row, dtype, w, G)
        assert (sg[b, g, :out_lo[b]] == -5.0).all() and (sg[b, g, out_hi[b]:] == -5.0).all()


@pytest.mark.parametrize("G", [4, 8])
def test_score_long_causal_window_matches_oracle(cuda_lib, G):
    """Several row chunks (w G > 256): causal skipping of key tiles (pass 1)
    and row chunks (pass 2) must not change any score.  Sequence 0 is a
    prompt scored against itself (positions ascending), sequence 1 a window
    of scattered positions in descending order."""
    se = cuda_lib
    B, Hkv, D, w, ctx = 2, 2, 128, 600, 1400
    dtype = torch.bfloat16
    shape = W.Shape(name="scl", B=B, Hq=Hkv * G, Hkv=Hkv, D=D, page_size=16, ctx=ctx, dtype=dtype)
    pc = W.build_paged_cache(shape, num_pages=B * 88 + 2, max_ctx=ctx, device="cuda", tag="scl")
    q_win = W.normal((B, w, shape.Hq, D), dtype, "cuda", "scl", "q", D, G)
    gen = torch.Generator().manual_seed(7)
    scattered = torch.randperm(ctx, generator=gen)[:w].sort(descending=True).values
    q_pos = torch.stack([torch.arange(ctx - w, ctx), scattered]).to(torch.int32)
    z, n = H.ranges(B, 0, ctx)
    scores = torch.full((B, Hkv, ctx), -5.0, device="cuda")
    se.se_score_window(se.kv_desc(pc, shape.Hq), q_win, q_pos.cuda(), z, n, z, n, causal=True,
                       accumulate=False, n_max=ctx, scores=scores)
    torch.cuda.synchronize()
    c = ocache.from_tensors(pc)
    os_ = oscore.score_window(c, q_win, q_pos.numpy(), [0] * B, [ctx] * B, [0] * B, [ctx] * B, True)
    sg = scores.cpu().double().numpy()
    for (b, g), row in os_.items():
        H.assert_scores_close(sg[b, g], row, dtype, w, G)


def test_score_window_accumulates(cuda_lib):
    se = cuda_lib
    B, Hkv, G, w, ctx = 1, 1, 4, 8, 100
    shape = W.Shape(name="sca", B=B, Hq=G, Hkv=Hkv, D=64, page_size=16, ctx=ctx, dtype=torch.float32)
    pc = W.build_paged_cache(shape, num_pages=8, max_ctx=ctx, device="cuda", tag="sca")
    q_win = W.normal((B, w, G, 64), torch.float32, "cuda", "sca")
    q_pos = torch.arange(ctx - w, ctx, dtype=torch.int32).cuda()[None]
    z, n = H.ranges(1, 0, ctx)
    scores = torch.ones((1, 1, ctx), device="cuda")
    for _ in range(2):
        se.se_score_window(se.kv_desc(pc, G), q_win, q_pos, z, n, z, n, causal=True,
                           accumulate=True, n_max=ctx, scores=scores)
    torch.cuda.synchronize()
    c = ocache.from_tensors(pc)
    row = oscore.score_window(c, q_win, q_pos.cpu().numpy(), [0], [ctx], [0], [ctx], True)[(0, 0)]
    H.assert_scores_close(scores[0, 0].cpu().double().numpy(), 1.0 + 2 * row, torch.float32, w, G)


def test_score_window_short_range_after_long_on_one_workspace(cuda_lib):
    """One row chunk (the persistent kernels) with far fewer key tiles than
    CTAs: 8 groups of 2 tiles (a 256-key range) under n_max = 4096, on a
    workspace that a 4096-key call has just used.  Pass 2 merges the pass-1
    slots of every CTA in a group's span, CTAs without tiles included; those
    must read as empty, not as the earlier call's statistics."""
    se = cuda_lib
    B, Hkv, G, w, ctx = 1, 8, 4, 64, 4096
    shape = W.Shape(name="scs", B=B, Hq=Hkv * G, Hkv=Hkv, D=128, page_size=16, ctx=ctx,
                    dtype=torch.bfloat16)
    pc = W.build_paged_cache(shape, num_pages=B * W.cdiv(ctx, 16) + 2, max_ctx=ctx, device="cuda",
                             tag="scs")
    q_win = W.normal((B, w, shape.Hq, 128), torch.bfloat16, "cuda", "scs", "q")
    kv = se.kv_desc(pc, shape.Hq)
    ws = torch.zeros(se._lib.se_score_window_workspace_size(kv, w, ctx), dtype=torch.uint8,
                     device="cuda")
    c = ocache.from_tensors(pc)
    for n in (ctx, 256):
        q_pos = torch.arange(n - w, n, dtype=torch.int32)[None].cuda()
        z, hi = H.ranges(B, 0, n)
        out = torch.full((B, Hkv, ctx), -5.0, device="cuda")
        se.se_score_window(kv, q_win, q_pos, z, hi, z, hi, causal=True, accumulate=False,
                           n_max=ctx, scores=out, workspace=ws)
        torch.cuda.synchronize()
        assert H.status(pc) == 0
        ref = oscore.score_window(c, q_win, q_pos.cpu().numpy(), [0], [n], [0], [n], True)
        sg = out.cpu().double().numpy()
        for (b, g), row in ref.items():
            H.assert_scores_close(sg[b, g, :n], row, torch.bfloat16, w, G)


@pytest.mark.parametrize("w", [64, 100])
def test_score_window_wait_limit_runs_out(cuda_lib, w):
    """The default (two-launch) tcgen05 scorer honours the wait limit in the
    workspace's control block: with 1 ns the key producer's first wait for a
    free stage gives up, the status word reads SE_ERR_TIMEOUT, the place is
    recorded and the launch winds down (the drains still wait for copies and
    MMAs in flight).  The next call on the same workspace (limit cleared,
    status reset) gives the scores of a call on a fresh workspace bit for bit
    and matches the oracle on a sampled group.  w = 64: one chunk of 256 rows
    (persistent kernels); w = 100: two row chunks (the grid kernels).  16384
    keys give every CTA more key tiles than its stage ring holds."""
    se = cuda_lib
    B, Hkv, G, ctx = 2, 4, 4, 16384
    tag = f"sto{w}"
    shape = W.Shape(name=tag, B=B, Hq=Hkv * G, Hkv=Hkv, D=128, page_size=16, ctx=ctx,
                    dtype=torch.bfloat16)
    pc = W.build_paged_cache(shape, num_pages=B * W.cdiv(ctx, 16) + 3, max_ctx=ctx, device="cuda",
                             tag=tag)
    q_win = W.normal((B, w, shape.Hq, 128), torch.bfloat16, "cuda", tag, "q")
    q_pos = torch.arange(ctx - w, ctx, dtype=torch.int32).repeat(B, 1).cuda()
    kv = se.kv_desc(pc, shape.Hq)
    nbytes = se._lib.se_score_window_workspace_size(kv, w, ctx)
    ws = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    z, n = H.ranges(B, 0, ctx)
    lo, hi = H.ranges(B, 0, ctx - w)

    def call(workspace):
        out = torch.zeros((B, Hkv, ctx), device="cuda")
        se.se_score_window(kv, q_win, q_pos, z, n, lo, hi, causal=True, accumulate=False,
                           n_max=ctx, scores=out, workspace=workspace)
        torch.cuda.synchronize()
        return out

    ws[:8].view(torch.int64).fill_(1)
    call(ws)
    assert H.status(pc) == se.SE_ERR_TIMEOUT
    assert int(ws[12:16].view(torch.int32).item()) != 0
    ws[:16].zero_()
    pc.status.zero_()
    again = call(ws)
    assert H.status(pc) == 0
    fresh = call(torch.zeros(nbytes, dtype=torch.uint8, device="cuda"))
    assert torch.equal(again, fresh)
    c = ocache.from_tensors(pc)
    ref = oscore.score_window(c, q_win, q_pos.cpu().numpy(), [0] * B, [ctx] * B, [0] * B,
                              [ctx - w] * B, True, groups=[(1, 3)])
    H.assert_scores_close(again[1, 3, :ctx - w].cpu().double().numpy(), ref[(1, 3)],
                          torch.bfloat16, w, G)
