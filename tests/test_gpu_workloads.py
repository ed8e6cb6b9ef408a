"""End-to-end GPU vs oracle on the five workloads.

Reduced sizes run the oracle over everything; the full sizes use the launch
configuration the benchmark times and check the oracle on sampled (sequence,
KV head) pairs / sequences, plus every integer result.  Inputs are the seeded
generators' only.
"""
import numpy as np
import pytest
import torch

import se_workloads as W
from attention_scored_sparse_gb300 import pipelines as P
from oracle import attention as oattn
from oracle import cache as ocache
from oracle import pipelines as opipe
from oracle import quest as oquest
from oracle import scoring as oscore
from oracle import selection as osel
from tests import gpu_helpers as H

pytestmark = pytest.mark.gpu


def _check_scores(scores_gpu, oracle_scores, lo_of_b, dtype, w, G):
    sg = scores_gpu.cpu().double().numpy()
    for (b, g), row in oracle_scores.items():
        lo = lo_of_b[b]
        H.assert_scores_close(sg[b, g, lo:lo + len(row)], row, dtype, w, G)


def _check_out(o_gpu, oracle_o, dtype, G):
    og = o_gpu.double().cpu().numpy()
    for (b, g), ref in oracle_o.items():
        err = np.abs(og[b, g * G:(g + 1) * G] - ref).max()
        assert err <= H.OUT_ATOL[dtype], (b, g, err)


# ---------------------------------------------------------------------------
# SnapKV
# ---------------------------------------------------------------------------


def _gpu_keep_after_ties(kg, ref_keep, rankings, k, forced):
    """The GPU's kept sets, each checked against the oracle's: equal, or
    different only at oracle near-ties of the k-th score (then the GPU's set
    is an equally valid answer and the later stages follow it).  Returns the
    kept lists and the number of (sequence, head) pairs that differed."""
    keep, resynced = [], 0
    for b in range(len(ref_keep)):
        kb = []
        for h in range(len(ref_keep[b])):
            d = H.assert_keep_near(kg[b, h], ref_keep[b][h], rankings[(b, h)], k, forced)
            resynced += d > 0
            kb.append(np.asarray(kg[b, h], dtype=np.int64))
        keep.append(kb)
    return keep, resynced


def _snapkv(cuda_lib, shape):
    """Scores element-wise, kept sets under the tie rule, then compaction and
    decode of the oracle on the kept sets the GPU chose (equal to the
    oracle's or differing only at near-ties): the cache bit for bit and the
    decode output always compared.  Returns the number of re-synchronised
    (sequence, KV head) pairs."""
    inp = W.snapkv_inputs(shape, "cuda")
    pc = inp["cache"]
    c = ocache.from_tensors(pc)
    ref = opipe.snapkv_select(c, inp["q_win"], inp["q_pos"].cpu().numpy(), shape)
    pipe = P.SnapKV(pc, shape.Hq, ctx=shape.ctx, window=shape.window, budget=shape.budget,
                    pool_kernel=shape.pool_kernel)
    o = torch.empty_like(inp["q_dec"])
    pipe.score(inp["q_win"], inp["q_pos"])
    pipe.select()
    torch.cuda.synchronize()
    _check_scores(pipe.scores, ref["scores"], [0] * shape.B, shape.dtype, shape.window, shape.G)
    rankings = {(b, h): H.pooled_scores(ref["scores"][(b, h)], 0, shape.pool_kernel)
                for b in range(shape.B) for h in range(shape.Hkv)}
    keep, resynced = _gpu_keep_after_ties(pipe.keep.cpu().numpy(), ref["keep"], rankings,
                                          shape.keep_topk, range(shape.scored, shape.ctx))
    o_ref = opipe.snapkv_finish(c, keep, inp["q_dec"])
    pipe.compact()
    pipe.decode(inp["q_dec"], o)
    torch.cuda.synchronize()
    assert H.status(pc) == 0
    H.assert_cache_equal(pc, c)
    _check_out(o, o_ref, shape.dtype, shape.G)
    assert (pc.ctx_len.cpu() == shape.budget).all()
    return resynced


def test_snapkv_tiny_workload(cuda_lib):
    assert _snapkv(cuda_lib, W.snapkv_tiny()) == 0


def test_snapkv_llama8b_reduced(cuda_lib):
    assert _snapkv(cuda_lib, W.snapkv_llama8b(B=2, ctx=4096 + 37, window=64, budget=512)) <= 2


@pytest.mark.parametrize("form", ["step", "two_streams"])
def test_snapkv_step_decodes_beside_compaction(cuda_lib, form):
    """The pipeline step (compaction and decode attention in one pass over the
    kept entries), and the form that runs decode attention on a second stream
    over the kept entries in their old pages while compaction moves them:
    the output equals, bit for bit, decode attention over the compacted
    cache, and the compacted cache is the one the separate calls leave."""
    shape = W.snapkv_llama8b(B=2, ctx=4096 + 37, window=64, budget=512)
    runs = []
    for overlapped in (False, True):
        inp = W.snapkv_inputs(shape, "cuda")
        pc = inp["cache"]
        pipe = P.SnapKV(pc, shape.Hq, ctx=shape.ctx, window=shape.window, budget=shape.budget,
                        pool_kernel=shape.pool_kernel)
        o = torch.full_like(inp["q_dec"], float("nan"))
        if overlapped and form == "step":
            pipe.step(inp["q_win"], inp["q_pos"], inp["q_dec"], o)
        elif overlapped:
            pipe.score(inp["q_win"], inp["q_pos"])
            pipe.select()
            pipe.compact_decode(inp["q_dec"], o)
        else:
            pipe.score(inp["q_win"], inp["q_pos"])
            pipe.select()
            pipe.compact()
            pipe.decode(inp["q_dec"], o)
        torch.cuda.synchronize()
        assert H.status(pc) == 0
        runs.append((o.clone(), {n: getattr(pc, n).clone() for n in
                                 ("block_table", "slot_map", "ctx_len", "free_list", "free_top",
                                  "k_pool", "v_pool")}))
    (o_seq, c_seq), (o_ovl, c_ovl) = runs
    assert torch.equal(o_seq, o_ovl)
    for n in c_seq:
        assert torch.equal(c_seq[n], c_ovl[n]), n


@pytest.mark.slow
def test_snapkv_llama8b_full(cuda_lib):
    """4 x 32768 tokens, 32/8 heads, budget 2048: full oracle (about 30 s).
    At most a few (sequence, KV head) pairs may follow a near-tie."""
    assert _snapkv(cuda_lib, W.snapkv_llama8b()) <= 4


# ---------------------------------------------------------------------------
# Quest
# ---------------------------------------------------------------------------


def _quest(cuda_lib, shape, steps, fused=False):
    """Page bounds' metadata bit for bit; per step the selected pages under
    the tie rule, then the oracle's attention over the pages the GPU chose
    (the oracle's own or a near-tie alternative) for every (sequence, head)."""
    inp = W.quest_inputs(shape, "cuda")
    pc = inp["cache"]
    c = ocache.from_tensors(pc)
    kmin, kmax = oquest.build_meta(c)
    pipe = P.QuestDecode(pc, shape.Hq, ctx=shape.ctx, top_pages=shape.top_pages)
    pipe.build_meta()
    nb = W.cdiv(shape.ctx, shape.page_size)
    torch.cuda.synchronize()
    for b in range(shape.B):
        pages = c.block_table[b, :nb]
        np.testing.assert_array_equal(pipe.kmin[pages].double().cpu().numpy(), kmin[pages])
        np.testing.assert_array_equal(pipe.kmax[pages].double().cpu().numpy(), kmax[pages])
    for t in steps:
        q = inp["q_steps"][t]
        o = torch.empty_like(q)
        pipe.page_idx.fill_(-7)
        (pipe.step_fused if fused else pipe.step)(q, o)
        torch.cuda.synchronize()
        ref = opipe.quest_select(c, kmin, kmax, q, shape.top_pages)
        got = pipe.page_idx.cpu().numpy()
        sel_gpu = {}
        for (b, g), sel in ref["sel"].items():
            U = ref["bounds"][(b, g)]
            ranking = {i: float(U[i]) for i in range(nb - 1)}
            row = got[b, g]
            n = len(sel)
            assert (row[n:] == -1).all(), (b, g, row)     # -1 after the selected pages
            H.assert_keep_near(row[:n], sel, ranking, min(shape.top_pages, nb - 1), [nb - 1])
            sel_gpu[(b, g)] = np.asarray(row[:n], dtype=np.int64)
        _check_out(o, opipe.quest_attend(c, q, sel_gpu), shape.dtype, shape.G)
    assert H.status(pc) == 0
    # Quest keeps the whole history resident
    assert (pc.ctx_len.cpu() == shape.ctx).all()


@pytest.mark.parametrize("fused", [False, True])
def test_quest_reduced(cuda_lib, fused):
    _quest(cuda_lib, W.quest_decode(ctx=16 * 700 + 5, top_pages=64, steps=3), range(3), fused)


@pytest.mark.parametrize("fused", [False, True])
def test_quest_fused_small_contexts(cuda_lib, fused):
    # fewer full pages than top_pages; a context inside the first page; G = 8
    _quest(cuda_lib, W.quest_decode(B=3, ctx=16 * 9 + 3, top_pages=20, steps=2), range(2), fused)
    _quest(cuda_lib, W.quest_decode(B=2, ctx=11, top_pages=4, steps=1), range(1), fused)
    _quest(cuda_lib, W.quest_decode(B=2, Hq=32, Hkv=4, ctx=16 * 300, top_pages=33, steps=1),
           range(1), fused)


@pytest.mark.slow
@pytest.mark.parametrize("fused", [False, True])
def test_quest_full(cuda_lib, fused):
    """2 x 131072 tokens, top 128 pages + current: steps 0 and 63 checked."""
    _quest(cuda_lib, W.quest_decode(), [0, 63], fused)


# ---------------------------------------------------------------------------
# H2O
# ---------------------------------------------------------------------------


def _h2o_lockstep(cuda_lib, shape, steps, seqs=None, data_every=1):
    """H2O end to end in lock-step with the oracle.

    Prompt: causal scores of the whole prompt (element-wise on the sampled
    sequences ``seqs``, every sequence by default), the kept sets under the
    tie rule, then the oracle's compaction on the kept sets the GPU chose --
    its own or a near-tie alternative -- bit for bit over every sequence.
    Decode: each step's output and running scores on the sampled sequences,
    their victims under the tie rule (a near-tie re-synchronises the oracle
    to the GPU's victim), and the cache's integer state (block table, slot
    maps, lengths, free list) of every sequence after every step; K/V bytes
    of the sampled sequences every step and of all every ``data_every``
    steps.  Sequences outside the sample follow the GPU's kept sets and
    victims, checked by their properties (count, order, forced range, the
    recent boundary).  Returns the number of re-synchronised choices."""
    inp = W.h2o_inputs(shape, "cuda", steps=steps)
    pc = inp["cache"]
    c = ocache.from_tensors(pc)
    B, Hkv, ctx = shape.B, shape.Hkv, shape.ctx
    sampled = list(range(B)) if seqs is None else list(seqs)
    groups = [(b, g) for b in sampled for g in range(Hkv)]
    acc_o = np.zeros(c.slot_map.shape)
    ref = opipe.h2o_prefill_select(c, inp["q_prompt"], inp["q_pos"].cpu().numpy(), shape, acc_o,
                                   groups=groups)
    pipe = P.H2O(pc, shape.Hq, prompt=ctx, heavy=shape.heavy, recent=shape.recent)
    pipe.prefill_score(inp["q_prompt"], inp["q_pos"])
    torch.cuda.synchronize()
    sg = pipe.acc[sampled].cpu().double().numpy()
    for i, b in enumerate(sampled):
        for g in range(Hkv):
            H.assert_scores_close(sg[i, g, :ctx], ref["scores"][(b, g)], shape.dtype, ctx, shape.G)
    pipe.prefill_select()
    torch.cuda.synchronize()
    kg = pipe.keep.cpu().numpy()
    recent = range(ctx - shape.recent, ctx)
    resynced = 0
    keep = []
    for b in range(B):
        kb = []
        for h in range(Hkv):
            if b in sampled:
                s_o = ref["scores"][(b, h)]
                ranking = {j: float(s_o[j]) for j in range(ctx - shape.recent)}
                resynced += H.assert_keep_near(kg[b, h], ref["keep"][b][h], ranking, shape.heavy,
                                               recent) > 0
            else:
                row = [int(x) for x in kg[b, h]]
                assert row == sorted(set(row)) and len(row) == shape.budget
                assert set(recent) <= set(row) and 0 <= row[0]
            kb.append(np.asarray(kg[b, h], dtype=np.int64))
        keep.append(kb)
    pipe.prefill_compact()
    assert ocache.compact(c, keep, [0] * B, aux=acc_o) == ocache.SE_OK
    torch.cuda.synchronize()
    assert H.status(pc) == 0
    H.assert_cache_equal(pc, c)
    np.testing.assert_allclose(pipe.acc[sampled].cpu().double().numpy(), acc_o[sampled],
                               rtol=1e-3, atol=1e-9)
    for t in range(steps):
        o = torch.empty_like(inp["q_steps"][t])
        pipe.step(inp["q_steps"][t], inp["k_steps"][t], inp["v_steps"][t], o)
        o_ref = opipe.h2o_step_attend(c, acc_o, inp["q_steps"][t], inp["k_steps"][t],
                                      inp["v_steps"][t], groups=groups)
        v_o = opipe.h2o_victims(c, acc_o, shape, seqs=sampled)
        torch.cuda.synchronize()
        assert H.status(pc) == 0
        vg = pipe.victim.cpu().numpy().astype(np.int64)
        for b in range(B):
            n = int(c.ctx_len[b])
            if b in sampled:
                for g in np.nonzero(vg[b] != v_o[b])[0]:
                    # only a near-tie of the oracle's running scores may differ
                    x, y = acc_o[b, g, vg[b, g]], acc_o[b, g, v_o[b, g]]
                    assert abs(x - y) <= H.TIE_REL * abs(y), (t, b, g, x, y)
                    resynced += 1
            elif n <= shape.budget:
                assert (vg[b] == -1).all(), (t, b)
            else:
                assert ((vg[b] >= 0) & (vg[b] < n)).all(), (t, b, vg[b])
                pos = c.slot_map[b, np.arange(Hkv), vg[b]]
                assert (pos < int(c.logical_len[b]) - shape.recent).all(), (t, b)
        assert ocache.move_last(c, vg, aux=acc_o) == ocache.SE_OK
        full = (t + 1) % data_every == 0 or t == steps - 1
        H.assert_cache_equal(pc, c, data_seqs=None if full else sampled)
        np.testing.assert_allclose(pipe.acc[sampled].cpu().double().numpy(), acc_o[sampled],
                                   rtol=1e-3, atol=1e-7)
        _check_out(o, o_ref, shape.dtype, shape.G)
    assert (pc.ctx_len.cpu() == shape.budget).all()
    return resynced


def test_h2o_reduced_lockstep(cuda_lib):
    shape = W.h2o_decode(B=3, ctx=300, heavy=100, recent=20, steps=40)
    assert _h2o_lockstep(cuda_lib, shape, 40) <= 2


@pytest.mark.slow
def test_h2o_full_end_to_end(cuda_lib):
    """The full H2O workload: 64 x 4096-token prompts compressed to 1024 +
    128, then 512 decode steps with evict-one; float results on sequences 0,
    31 and 63, integer state of all 64 after every step."""
    shape = W.h2o_decode()
    assert _h2o_lockstep(cuda_lib, shape, shape.steps, seqs=[0, 31, 63], data_every=64) <= 8


def test_h2o_full_decode_lockstep_from_generated_state(cuda_lib):
    """64 sequences at the steady-state budget (1152 resident + the new token),
    full-size decode steps in lock-step from one generated state."""
    shape = W.h2o_decode(ctx=1152)
    steps = 3
    inp = W.h2o_inputs(shape, "cuda", steps=steps)
    pc = inp["cache"]
    c = ocache.from_tensors(pc)
    acc = torch.rand(c.slot_map.shape, generator=W.generator("cpu", "h2o_acc")).cuda() * 10
    acc_o = acc.double().cpu().numpy()
    pipe = P.H2O(pc, shape.Hq, prompt=1152, heavy=shape.heavy, recent=shape.recent)
    pipe.acc.copy_(acc)
    for t in range(steps):
        o = torch.empty_like(inp["q_steps"][t])
        pipe.step(inp["q_steps"][t], inp["k_steps"][t], inp["v_steps"][t], o)
        r = opipe.h2o_step(c, acc_o, inp["q_steps"][t], inp["k_steps"][t], inp["v_steps"][t], shape)
        torch.cuda.synchronize()
        assert H.status(pc) == 0
        assert (pipe.victim.cpu().numpy() == r["victim"]).all()
        H.assert_cache_equal(pc, c, seqs=[0, 31, 63])
        np.testing.assert_allclose(pipe.acc.cpu().double().numpy(), acc_o, rtol=1e-5, atol=1e-6)
        _check_out(o, r["o"], shape.dtype, shape.G)


def _h2o_chunked(cuda_lib, shape, chunk):
    """Chunk-wise prefill eviction in lock-step with the oracle: running
    scores after every chunk, the kept sets (near-ties of the oracle's k-th
    score re-synchronised to the GPU's choice) and the cache bit for bit."""
    inp = W.h2o_chunked_inputs(shape, chunk, "cuda")
    pc = inp["cache"]
    c = ocache.from_tensors(pc)
    acc_o = np.zeros(c.slot_map.shape)
    pipe = P.H2OChunkedPrefill(pc, shape.Hq, chunk=chunk, heavy=shape.heavy, recent=shape.recent)
    resident, resynced = 0, 0
    for i in range(inp["q_chunks"].shape[0]):
        ctx = resident + chunk
        resident = pipe.chunk_step(resident, inp["q_chunks"][i], inp["q_pos"][i],
                                   inp["k_chunks"][i], inp["v_chunks"][i])
        torch.cuda.synchronize()
        assert H.status(pc) == 0
        assert ocache.append_tokens(c, ocache._bits(inp["k_chunks"][i]),
                                    ocache._bits(inp["v_chunks"][i]), aux=acc_o) == ocache.SE_OK
        s = oscore.score_window(c, inp["q_chunks"][i], inp["q_pos"][i].cpu().numpy(),
                                [0] * shape.B, [ctx] * shape.B, [0] * shape.B, [ctx] * shape.B, True)
        for (b, h), v in s.items():
            acc_o[b, h, :ctx] += v
        if ctx > shape.budget:
            kg = pipe.keep.cpu().numpy()
            keep = []
            for b in range(shape.B):
                kb = []
                for h in range(shape.Hkv):
                    ko = osel.topk_keep(acc_o[b, h, :ctx - shape.recent], 0, shape.heavy, 1,
                                        ctx - shape.recent, ctx)
                    ranking = {j: float(acc_o[b, h, j]) for j in range(ctx - shape.recent)}
                    resynced += H.assert_keep_near(kg[b, h], ko, ranking, shape.heavy,
                                                   range(ctx - shape.recent, ctx))
                    kb.append(kg[b, h].astype(np.int64))     # follow the GPU (equal or a near-tie)
                keep.append(kb)
            assert ocache.compact(c, keep, [0] * shape.B, aux=acc_o) == ocache.SE_OK
        H.assert_cache_equal(pc, c)
        n = int(c.ctx_len[0])
        np.testing.assert_allclose(pipe.acc[:, :, :n].cpu().double().numpy(), acc_o[:, :, :n],
                                   rtol=2e-3, atol=1e-6)
        acc_o[:, :, :n] = pipe.acc[:, :, :n].cpu().double().numpy()   # no drift between chunks
    assert resident == min(shape.budget, shape.ctx)
    return resynced


def test_h2o_chunked_prefill_reduced(cuda_lib):
    shape = W.h2o_decode(B=2, Hq=8, Hkv=2, ctx=1024, heavy=192, recent=64)
    _h2o_chunked(cuda_lib, shape, 256)


def test_h2o_chunked_prefill_ragged_pages(cuda_lib):
    # budget and chunk not multiples of the page size
    shape = W.h2o_decode(B=3, Hq=8, Hkv=2, ctx=600, heavy=101, recent=23)
    _h2o_chunked(cuda_lib, shape, 120)


def _kara_schedule(cuda_lib, shape, steps):
    """Kara compression inside a decode loop, staggered over the batch, in
    lock-step with the oracle: the cache bit for bit after every step, kept
    sets of every compression, attention outputs."""
    inp = W.kara_schedule_inputs(shape, "cuda", steps=steps)
    pc = inp["cache"]
    c = ocache.from_tensors(pc)
    fills = [shape.fill(b) for b in range(shape.B)]
    ring_g = inp["q_ring"].clone()
    ring_o = inp["q_ring"].cpu().clone()
    win_start = [shape.ctx - f for f in fills]
    pipe = P.KaraSchedule(pc, shape.Hq, ctx=shape.ctx, fills=fills, window=shape.window,
                          protected=shape.protected, candidates=shape.candidates,
                          budget=shape.budget, chunk_coef=shape.chunk_coef,
                          max_ctx=shape.ctx + steps)
    n_due = 0
    for t in range(steps):
        o = torch.empty_like(inp["q_steps"][t])
        due = pipe.step(inp["q_steps"][t], inp["k_steps"][t], inp["v_steps"][t], o, ring_g)
        r = opipe.kara_schedule_step(c, inp["q_steps"][t].cpu(), inp["k_steps"][t].cpu(),
                                     inp["v_steps"][t].cpu(), ring_o, win_start, shape)
        torch.cuda.synchronize()
        assert H.status(pc) == 0
        assert due == r["due"], (t, due, r["due"])
        n_due += len(due)
        if due:
            kg = pipe.keep.cpu().numpy()
            for b in due:
                for h in range(shape.Hkv):
                    assert list(kg[b, h]) == list(r["keep"][b][h]), (t, b, h)
        H.assert_cache_equal(pc, c)
        _check_out(o, r["o"], shape.dtype, shape.G)
    assert n_due >= shape.B
    return n_due


def test_kara_schedule_reduced(cuda_lib):
    shape = W.kara_schedule(B=5, Hq=8, Hkv=2, ctx=300, window=64, protected=8, candidates=8,
                            budget=16)
    _kara_schedule(cuda_lib, shape, 90)


# ---------------------------------------------------------------------------
# Kara + prune
# ---------------------------------------------------------------------------


def _kara(cuda_lib, shape, seqs=None):
    inp = W.kara_inputs(shape, "cuda")
    pc = inp["cache"]
    nb = shape.ctx // shape.page_size
    c = ocache.from_tensors(pc, seqs=seqs, blocks=(nb - shape.window // shape.page_size, nb)) \
        if seqs is not None else ocache.from_tensors(pc)
    ref = opipe.kara_compress(c, inp["q_win"], inp["q_pos"].cpu().numpy(), shape)
    pipe = P.Kara(pc, shape.Hq, ctx=shape.ctx, window=shape.window, protected=shape.protected,
                  candidates=shape.candidates, budget=shape.budget, chunk_coef=shape.chunk_coef)
    pipe.score(inp["q_win"], inp["q_pos"])
    pipe.select()
    torch.cuda.synchronize()
    win_lo = shape.ctx - shape.window
    _check_scores(pipe.scores, ref["scores"], [win_lo] * shape.B, shape.dtype, shape.window, shape.G)
    kg = pipe.keep.cpu().numpy()
    for b in range(shape.B):
        for h in range(shape.Hkv):
            assert list(kg[b, h]) == list(ref["keep"][b][h]), (b, h)
    assert ocache.compact(c, ref["keep"], ref["first_slot"], seqs=seqs) == ocache.SE_OK
    pipe.compact()
    torch.cuda.synchronize()
    assert H.status(pc) == 0
    H.assert_cache_equal(pc, c, seqs=seqs)
    B = shape.B
    L = [shape.prune_L] * B
    R = [shape.prune_R] * B
    mask = inp["prune_mask"].cpu().numpy()
    st, busy = ocache.prune(c, L, R, mask, seqs=seqs)
    assert st == ocache.SE_OK
    pipe.prune(torch.tensor(L, dtype=torch.int32, device="cuda"),
               torch.tensor(R, dtype=torch.int32, device="cuda"), inp["prune_mask"])
    torch.cuda.synchronize()
    assert H.status(pc) == 0
    H.assert_cache_equal(pc, c, seqs=seqs)
    assert pipe.n_busy.cpu().tolist() == busy
    # logical prefix untouched, R' = (R \ T) U I
    assert (pc.logical_len.cpu() == shape.ctx).all()
    new_ctx = shape.prune_L + shape.prune_keep + (shape.ctx - shape.window - shape.prune_R) + \
        shape.budget + shape.protected
    assert (pc.ctx_len.cpu() == new_ctx).all()
    o = torch.empty_like(inp["q_dec"])
    pipe.decode(inp["q_dec"], o, max_entries=new_ctx)
    torch.cuda.synchronize()
    groups = None if seqs is None else [(b, g) for b in seqs for g in range(shape.Hkv)]
    oo, _ = oattn.decode_attention(c, opipe.to_f64(inp["q_dec"]), "dense", groups=groups)
    _check_out(o, oo, shape.dtype, shape.G)


def test_kara_reduced(cuda_lib):
    _kara(cuda_lib, W.kara_prune(B=4, ctx=2048 + 256, prune_L=256 + 7, prune_R=1024 + 3))


@pytest.mark.slow
def test_kara_full_sampled(cuda_lib):
    """128 x 16384 tokens: every score / keep / integer result of all
    sequences, K/V bytes and decode outputs on sampled sequences."""
    _kara(cuda_lib, W.kara_prune(), seqs=[0, 77, 127])
