"""Pins of the CPU oracle to facts that do not come from the oracle itself.

Each pin uses an independent source: torch library routines (scaled dot
product attention with V = I gives the attention probabilities, avg_pool1d),
Python's ``sorted`` as a brute-force ranking, closed forms, invariants of the
page accounting, and hand-worked fixtures under tests/golden/.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import attention, cache, pipelines, quest, scoring, selection
from oracle.cache import values
import se_workloads as W
from tests.helpers import sdpa_out, sdpa_probs, tiny_cache, tiny_shape

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def oc(pc):
    return cache.from_tensors(pc)


# ---------------------------------------------------------------------------
# O1 window scoring
# ---------------------------------------------------------------------------


def _set_identical_keys(pc):
    """Every resident key of head h equal to one vector (per head)."""
    for h in range(pc.Hkv):
        kvec = torch.arange(pc.D, dtype=torch.float32) * 0.25 - 1.0 + h
        pc.k_pool[:, h, :, :] = kvec.to(pc.k_pool.dtype)


def test_scores_identical_keys_causal_closed_form():
    # equal logits: each row spreads 1/(#visible) over its visible keys; a
    # query at position t sees t+1 keys, so s_j = G * sum_{t_q >= j} 1/(t_q+1)
    shape = tiny_shape(ctx=22)
    pc = tiny_cache(shape)
    _set_identical_keys(pc)
    c = oc(pc)
    w = 6
    q = torch.randn(shape.B, w, shape.Hq, shape.D, generator=W.generator("cpu", "pin", "q"))
    q_pos = np.tile(np.arange(shape.ctx - w, shape.ctx), (shape.B, 1))
    s = scoring.score_window(c, q.numpy(), q_pos, [0] * 2, [22] * 2, [0] * 2, [22] * 2, True)
    G = shape.G
    for (b, g), sv in s.items():
        for j in range(22):
            expect = G * sum(1.0 / (t + 1) for t in q_pos[b] if t >= j)
            assert sv[j] == pytest.approx(expect, rel=1e-12)


def test_scores_identical_keys_bidirectional_closed_form():
    shape = tiny_shape(ctx=20)
    pc = tiny_cache(shape)
    _set_identical_keys(pc)
    c = oc(pc)
    w = 8
    q = torch.randn(shape.B, w, shape.Hq, shape.D, generator=W.generator("cpu", "pin", "qb"))
    q_pos = np.tile(np.arange(12, 20), (shape.B, 1))
    s = scoring.score_window(c, q.numpy(), q_pos, [12] * 2, [20] * 2, [12] * 2, [18] * 2, False)
    for sv in s.values():
        np.testing.assert_allclose(sv, shape.G * w / 8, rtol=1e-12)


@pytest.mark.parametrize("causal", [True, False])
def test_scores_match_library_attention_probabilities(causal):
    # torch SDPA with V = identity returns the softmax matrix; its column sums
    # over the group's heads and window queries are the scores
    shape = tiny_shape(ctx=26, D=16)
    pc = tiny_cache(shape)
    c = oc(pc)
    w = 5
    q = torch.randn(shape.B, w, shape.Hq, shape.D, generator=W.generator("cpu", "pin", "ql"))
    q_pos = np.tile(np.arange(21, 26), (shape.B, 1))
    lo, hi, olo, ohi = 3, 26, 4, 21
    s = scoring.score_window(c, q.numpy(), q_pos, [lo] * 2, [hi] * 2, [olo] * 2, [ohi] * 2, causal)
    for b in range(shape.B):
        for g in range(shape.Hkv):
            K = c.keys(b, g, range(lo, hi))
            pos = c.slot_map[b, g, lo:hi]
            total = np.zeros(hi - lo)
            for h in range(g * shape.G, (g + 1) * shape.G):
                Q = q[b, :, h, :].double().numpy()
                mask = (pos[None, :] <= q_pos[b][:, None]) if causal else None
                total += sdpa_probs(Q, K, mask).sum(axis=0)
            np.testing.assert_allclose(s[(b, g)], total[olo - lo: ohi - lo], rtol=1e-12, atol=1e-15)


def test_scores_rows_sum_to_one_and_single_key():
    shape = tiny_shape(ctx=18)
    pc = tiny_cache(shape)
    c = oc(pc)
    w = 4
    q = torch.randn(shape.B, w, shape.Hq, shape.D, generator=W.generator("cpu", "pin", "qr")) * 3
    q_pos = np.tile(np.arange(14, 18), (shape.B, 1))
    s = scoring.score_window(c, q.numpy(), q_pos, [0] * 2, [18] * 2, [0] * 2, [18] * 2, True)
    for sv in s.values():
        assert sv.sum() == pytest.approx(w * shape.G, rel=1e-12)
    s1 = scoring.score_window(c, q.numpy(), q_pos, [5] * 2, [6] * 2, [5] * 2, [6] * 2, False)
    for sv in s1.values():
        assert sv[0] == pytest.approx(w * shape.G, rel=1e-12)


def test_scores_causal_masks_future_keys():
    shape = tiny_shape(ctx=20)
    c = oc(tiny_cache(shape))
    q = torch.randn(shape.B, 3, shape.Hq, shape.D, generator=W.generator("cpu", "pin", "qf"))
    q_pos = np.tile(np.array([10, 11, 12]), (shape.B, 1))
    s = scoring.score_window(c, q.numpy(), q_pos, [0] * 2, [20] * 2, [0] * 2, [20] * 2, True)
    for sv in s.values():
        assert (sv[13:] == 0).all() and (sv[:13] > 0).all()


# ---------------------------------------------------------------------------
# O2 pooling
# ---------------------------------------------------------------------------


def test_pool_golden_hand_example():
    g = golden("pool7_len8.json")
    np.testing.assert_allclose(scoring.avg_pool(np.array(g["x"], float), g["kernel"]), g["expected"])


def test_pool_matches_library_avg_pool1d():
    x = torch.randn(97, generator=W.generator("cpu", "pin", "pool"), dtype=torch.float64)
    lib = torch.nn.functional.avg_pool1d(x[None, None], 7, stride=1, padding=3,
                                         count_include_pad=True)[0, 0].numpy()
    np.testing.assert_allclose(scoring.avg_pool(x.numpy(), 7), lib, rtol=1e-14)
    np.testing.assert_array_equal(scoring.avg_pool(x.numpy(), 1), x.numpy())


def test_pool_constant_input():
    out = scoring.avg_pool(np.full(20, 2.0), 7)
    np.testing.assert_allclose(out[3:17], 2.0)
    np.testing.assert_allclose(out[:3], [8 / 7, 10 / 7, 12 / 7])
    np.testing.assert_allclose(out[17:], [12 / 7, 10 / 7, 8 / 7])


# ---------------------------------------------------------------------------
# O3 top-k with forced ranges
# ---------------------------------------------------------------------------


@pytest.mark.parametrize("seed", range(5))
def test_topk_brute_force(seed):
    rng = np.random.default_rng(seed)
    n, k = 40, 9
    s = np.round(rng.random(n), 1)            # many ties
    keep = selection.topk_keep(s, 10, k, 1, 45, 50)
    cands = [j for j in range(10, 10 + n) if not 45 <= j < 50]   # forced slots are no candidates
    ranked = sorted(cands, key=lambda j: (-s[j - 10], j))[:k]
    assert list(keep) == sorted(ranked + list(range(45, 50)))


def test_topk_with_pool_brute_force():
    rng = np.random.default_rng(7)
    s = rng.random(60)
    pooled = torch.nn.functional.avg_pool1d(torch.tensor(s)[None, None], 7, 1, 3)[0, 0].numpy()
    keep = selection.topk_keep(s, 0, 12, 7, 60, 64)
    ranked = sorted(range(60), key=lambda j: (-pooled[j], j))[:12]
    assert list(keep) == sorted(ranked) + [60, 61, 62, 63]


def test_topk_window_sum_ranks_as_window_mean():
    """The device ranks pooled candidates by the zero-padded window sum; the
    pages define the window mean.  Dividing by the fixed width keeps the order,
    so the kept slots are the same (window sums taken here by convolution)."""
    rng = np.random.default_rng(11)
    for n, k, pool in [(200, 31, 7), (64, 10, 3), (129, 1, 5)]:
        s = rng.random(n)
        sums = np.convolve(s, np.ones(pool), mode="same")
        ranked = sorted(range(n), key=lambda j: (-sums[j], j))[:k]
        keep = selection.topk_keep(s, 0, k, pool, n, n)
        assert list(keep) == sorted(ranked)


def test_topk_all_equal_keeps_lowest_and_forced_overlap():
    keep = selection.topk_keep(np.ones(30), 0, 5, 1, 30, 32)
    assert list(keep) == [0, 1, 2, 3, 4, 30, 31]
    # a forced range inside the candidate range is not a candidate
    keep = selection.topk_keep(np.ones(30), 0, 5, 1, 2, 4)
    assert list(keep) == [0, 1, 2, 3, 4, 5, 6]


# ---------------------------------------------------------------------------
# O4 Kara Token2Chunk
# ---------------------------------------------------------------------------


def test_kara_golden_hand_example():
    g = golden("kara_token2chunk_hand.json")
    keep = selection.kara_keep(np.array(g["scores"]), g["cand_lo"], g["n_cand"], g["budget"],
                               g["coef"], g["force_lo"], g["force_hi"])
    assert list(keep) == g["expected"]


@pytest.mark.parametrize("seed", range(20))
def test_kara_invariants(seed):
    rng = np.random.default_rng(100 + seed)
    n, n_cand, budget = 224, 32, 64
    s = rng.random(n) * rng.choice([1.0, 10.0])
    keep = selection.kara_keep(s, 1000, n_cand, budget, 0.01, 1224, 1256)
    body = keep[:-32]
    assert list(keep[-32:]) == list(range(1224, 1256))
    assert len(body) == budget and (np.diff(body) > 0).all()
    top = sorted(range(n), key=lambda j: (-s[j], j))[:n_cand]
    assert set(1000 + j for j in top) <= set(body)


def test_kara_contiguous_candidates_reduce_to_topk():
    # if the top candidates are contiguous every chunk interior is empty and
    # the retained set is the top-`budget` by score (brute-force sorted)
    rng = np.random.default_rng(3)
    s = rng.random(224)
    s[50:82] += 10.0                      # 32 contiguous best tokens
    keep = selection.kara_keep(s, 0, 32, 64, 0.01, 224, 256)[:-32]
    ranked = sorted(range(224), key=lambda j: (-s[j], j))[:64]
    assert list(keep) == sorted(ranked)


def _kara_tiny():
    shape = W.kara_prune(B=2, Hq=4, Hkv=2, D=16, page_size=4, ctx=64, window=16, protected=4,
                         candidates=4, budget=6, prune_L=8, prune_R=24, dtype=torch.float32,
                         name="kara_pin")
    return shape, W.kara_inputs(shape, "cpu")


def test_kara_compress_identical_keys_softmax_spans_the_whole_window():
    # KARA Method 1: every window query attends to every window key, the
    # protected tail included; only the compressible columns are scored.
    # With one key vector per head each row gives 1/window to every window
    # key, so each compressible score is G * w / window -- and G * w /
    # (window - protected) if the protected keys were left out of the softmax.
    shape, inp = _kara_tiny()
    pc = inp["cache"]
    _set_identical_keys(pc)
    c = oc(pc)
    r = pipelines.kara_compress(c, inp["q_win"], inp["q_pos"].numpy(), shape)
    win_lo = shape.ctx - shape.window
    assert r["first_slot"] == [win_lo] * shape.B
    for (b, h), sv in r["scores"].items():
        assert len(sv) == shape.compressible
        np.testing.assert_allclose(sv, shape.G * shape.window / shape.window, rtol=1e-12)
        # all scores tie: the candidates are the lowest compressible slots,
        # contiguous, so no chunk has an interior and the top-up takes the
        # next lowest slots; the protected tail follows
        expect = list(range(win_lo, win_lo + shape.budget)) + \
            list(range(shape.ctx - shape.protected, shape.ctx))
        assert list(r["keep"][b][h]) == expect


def test_kara_compress_scores_are_library_attention_over_the_window():
    # column sums of torch SDPA probabilities (V = I) over the full window,
    # no mask, restricted to the compressible columns; the kept set is
    # Token2Chunk of those scores over [win_lo, ctx - protected) plus the tail
    shape, inp = _kara_tiny()
    c = oc(inp["cache"])
    r = pipelines.kara_compress(c, inp["q_win"], inp["q_pos"].numpy(), shape)
    win_lo, prot_lo = shape.ctx - shape.window, shape.ctx - shape.protected
    for b in range(shape.B):
        for g in range(shape.Hkv):
            K = c.keys(b, g, range(win_lo, shape.ctx))
            total = np.zeros(shape.window)
            for h in range(g * shape.G, (g + 1) * shape.G):
                total += sdpa_probs(inp["q_win"][b, :, h, :].double().numpy(), K).sum(axis=0)
            want = total[: prot_lo - win_lo]
            np.testing.assert_allclose(r["scores"][(b, g)], want, rtol=1e-12, atol=1e-15)
            # the protected columns carry real probability mass, so leaving them
            # out of the softmax would change every score above
            assert total[prot_lo - win_lo:].sum() > 1e-3 * total.sum()
            kept = selection.kara_keep(want, win_lo, shape.candidates, shape.budget,
                                       shape.chunk_coef, prot_lo, shape.ctx)
            assert list(r["keep"][b][g]) == list(kept)


# ---------------------------------------------------------------------------
# O5 H2O
# ---------------------------------------------------------------------------


@pytest.mark.parametrize("seed", range(5))
def test_h2o_victim_brute_force(seed):
    rng = np.random.default_rng(seed)
    ctx = 30
    acc = np.round(rng.random(40), 1)
    pos = rng.permutation(100)[:40]
    v = selection.h2o_victim(acc, pos, ctx, 29, 70)
    elig = [j for j in range(ctx) if pos[j] < 70]
    expect = sorted(elig, key=lambda j: (acc[j], -pos[j]))[0]
    assert v == expect
    assert selection.h2o_victim(acc, pos, ctx, 30, 70) == -1


def _h2o_tiny(budget_heavy, recent, steps, prompt=24):
    shape = W.h2o_decode(B=2, Hq=4, Hkv=2, D=16, ctx=prompt, heavy=budget_heavy, recent=recent,
                         steps=steps, dtype=torch.float32, name="h2o_tiny")
    inp = W.h2o_inputs(shape, "cpu")
    return shape, inp


def test_h2o_pipeline_invariants_and_acc_recomputation():
    shape, inp = _h2o_tiny(8, 4, 10)
    c = oc(inp["cache"])
    orig = c.copy()
    acc = np.zeros(c.slot_map.shape)
    pipelines.h2o_prefill(c, inp["q_prompt"], inp["q_pos"].numpy(), shape, acc)
    assert (c.ctx_len == shape.budget).all()
    # independent running score per logical position, from library attention
    run = {}
    for b in range(c.B):
        for g in range(c.Hkv):
            K = orig.keys(b, g, range(shape.ctx))
            tot = np.zeros(shape.ctx)
            for h in range(g * shape.G, (g + 1) * shape.G):
                Q = inp["q_prompt"][b, :, h].double().numpy()
                mask = np.arange(shape.ctx)[None, :] <= np.arange(shape.ctx)[:, None]
                tot += sdpa_probs(Q, K, mask).sum(axis=0)
            run[(b, g)] = {p: tot[p] for p in range(shape.ctx)}
    for t in range(shape.steps):
        pipelines.h2o_step(c, acc, inp["q_steps"][t], inp["k_steps"][t], inp["v_steps"][t], shape)
        for b in range(c.B):
            L = int(c.logical_len[b])
            assert c.ctx_len[b] == shape.budget
            for g in range(c.Hkv):
                pos = c.slot_map[b, g, : c.ctx_len[b]]
                assert set(range(L - shape.recent, L)) <= set(pos.tolist())
    # recompute acc for the survivors: prompt score + every step's group sum,
    # replaying each step's attention with library SDPA over the entries that
    # were resident at that step
    c2 = oc(inp["cache"])
    acc2 = np.zeros(c2.slot_map.shape)
    pipelines.h2o_prefill(c2, inp["q_prompt"], inp["q_pos"].numpy(), shape, acc2)
    for t in range(shape.steps):
        kb, vb = cache._bits(inp["k_steps"][t]), cache._bits(inp["v_steps"][t])
        cache.append(c2, kb, vb, aux=acc2)
        q = inp["q_steps"][t].double().numpy()
        for b in range(c2.B):
            for g in range(c2.Hkv):
                slots = np.arange(c2.ctx_len[b])
                K, pos = c2.keys(b, g, slots), c2.slot_map[b, g, slots]
                p = sum(sdpa_probs(q[b, h][None], K)[0] for h in range(g * shape.G, (g + 1) * shape.G))
                for j, pp in zip(pos, p):
                    run[(b, g)][int(j)] = run[(b, g)].get(int(j), 0.0) + pp
        # same evictions as the oracle run (positions), to stay in lock-step
        o, _ = attention.decode_attention(c2, q, "dense")
        for (b, g), (slots, pp) in _.items():
            acc2[b, g, slots] += pp
        victim = np.full((c2.B, c2.Hkv), -1)
        for b in range(c2.B):
            for g in range(c2.Hkv):
                victim[b, g] = selection.h2o_victim(acc2[b, g], c2.slot_map[b, g], int(c2.ctx_len[b]),
                                                    shape.budget, int(c2.logical_len[b]) - shape.recent)
        cache.move_last(c2, victim, aux=acc2)
    for b in range(c.B):
        for g in range(c.Hkv):
            for s in range(c.ctx_len[b]):
                assert acc[b, g, s] == pytest.approx(run[(b, g)][int(c.slot_map[b, g, s])], rel=1e-10)


def test_h2o_no_eviction_when_budget_covers_context():
    shape, inp = _h2o_tiny(100, 8, 4)
    c = oc(inp["cache"])
    acc = np.zeros(c.slot_map.shape)
    pipelines.h2o_prefill(c, inp["q_prompt"], inp["q_pos"].numpy(), shape, acc)
    for t in range(shape.steps):
        r = pipelines.h2o_step(c, acc, inp["q_steps"][t], inp["k_steps"][t], inp["v_steps"][t], shape)
        assert (r["victim"] == -1).all()
        for b in range(c.B):
            for g in range(c.Hkv):
                slots = np.arange(c.ctx_len[b])
                assert list(c.slot_map[b, g, slots]) == list(range(shape.ctx + t + 1))
                q = inp["q_steps"][t][b, g * shape.G:(g + 1) * shape.G].double().numpy()
                ref = sdpa_out(q, c.keys(b, g, slots), c.vals(b, g, slots))
                np.testing.assert_allclose(r["o"][(b, g)], ref, rtol=1e-12, atol=1e-14)


def _h2o_chunked_tiny(heavy, recent, prompt=48):
    shape = W.h2o_decode(B=2, Hq=4, Hkv=2, D=16, ctx=prompt, heavy=heavy, recent=recent,
                         steps=1, dtype=torch.float32, name="h2o_chunked_tiny")
    return shape, W.h2o_chunked_inputs(shape, 8, "cpu")


def _chunk_group_probs(inp, i, b, g, G, K, k_pos):
    """Library attention of chunk i's queries of group g over keys K (fp64)."""
    tot = np.zeros(K.shape[0])
    qpos = inp["q_pos"][i, b].numpy()
    mask = k_pos[None, :] <= qpos[:, None]
    for h in range(g * G, (g + 1) * G):
        Q = inp["q_chunks"][i, b, :, h].double().numpy()
        tot += sdpa_probs(Q, K, mask).sum(axis=0)
    return tot


def test_h2o_chunked_prefill_without_eviction_is_whole_prompt_scoring():
    """Budget above the prompt: chunks only split the queries, so the running
    scores are the causal column sums of the whole prompt (library SDPA)."""
    shape, inp = _h2o_chunked_tiny(100, 8)
    c = oc(inp["cache"])
    acc = np.zeros(c.slot_map.shape)
    for i in range(inp["q_chunks"].shape[0]):
        r = pipelines.h2o_prefill_chunk(c, acc, inp["q_chunks"][i], inp["q_pos"][i].numpy(),
                                        inp["k_chunks"][i], inp["v_chunks"][i], 100, 8)
        assert r["keep"] is None
    assert (c.ctx_len == shape.ctx).all() and (c.logical_len == shape.ctx).all()
    n_ch = inp["q_chunks"].shape[0]
    for b in range(c.B):
        for g in range(c.Hkv):
            slots = np.arange(shape.ctx)
            assert list(c.slot_map[b, g, slots]) == list(range(shape.ctx))
            K = values(cache._bits(inp["k_chunks"][:, b, :, g]).reshape(shape.ctx, shape.D))
            assert (c.keys(b, g, slots) == K).all()
            want = sum(_chunk_group_probs(inp, i, b, g, shape.G, K, slots) for i in range(n_ch))
            np.testing.assert_allclose(acc[b, g, :shape.ctx], want, rtol=1e-12, atol=1e-14)


def test_h2o_chunked_prefill_eviction_replayed_independently():
    """With eviction: replay every chunk with library attention over the
    entries resident at that chunk, keep per logical position a running score,
    and pick the survivors by a full sort; the oracle must agree at every
    chunk, keep the recent tokens and hold exactly heavy + recent entries."""
    heavy, recent = 12, 4
    shape, inp = _h2o_chunked_tiny(heavy, recent)
    c = oc(inp["cache"])
    before = c.copy()
    acc = np.zeros(c.slot_map.shape)
    G, chunk = shape.G, inp["q_chunks"].shape[2]
    run = {(b, g): {} for b in range(c.B) for g in range(c.Hkv)}      # position -> score
    keyv = {}                                                         # (b, g, position) -> key
    for i in range(inp["q_chunks"].shape[0]):
        for b in range(c.B):
            for g in range(c.Hkv):
                for j in range(chunk):
                    p = i * chunk + j
                    keyv[(b, g, p)] = values(cache._bits(inp["k_chunks"][i, b, j, g]))
                    run[(b, g)][p] = 0.0
                pos = np.array(sorted(run[(b, g)]))
                K = np.stack([keyv[(b, g, int(p))] for p in pos])
                probs = _chunk_group_probs(inp, i, b, g, G, K, pos)
                for p, v in zip(pos, probs):
                    run[(b, g)][int(p)] += v
                if len(pos) > heavy + recent:
                    old = pos[:-recent]
                    top = sorted(old, key=lambda p: (-run[(b, g)][int(p)], p))[:heavy]
                    survivors = set(int(p) for p in top) | set(int(p) for p in pos[-recent:])
                    run[(b, g)] = {p: run[(b, g)][p] for p in survivors}
        pipelines.h2o_prefill_chunk(c, acc, inp["q_chunks"][i], inp["q_pos"][i].numpy(),
                                    inp["k_chunks"][i], inp["v_chunks"][i], heavy, recent)
        _check_accounting(before, c)
        for b in range(c.B):
            n = int(c.ctx_len[b])
            assert n == min(heavy + recent, (i + 1) * chunk)
            for g in range(c.Hkv):
                pos = c.slot_map[b, g, :n]
                assert (np.diff(pos) > 0).all()
                assert sorted(run[(b, g)]) == pos.tolist()
                assert set(range((i + 1) * chunk - recent, (i + 1) * chunk)) <= set(pos.tolist())
                want = np.array([run[(b, g)][int(p)] for p in pos])
                np.testing.assert_allclose(acc[b, g, :n], want, rtol=1e-12, atol=1e-14)
                for s, p in enumerate(pos):
                    assert (c.keys(b, g, [s])[0] == keyv[(b, g, int(p))]).all()


def test_append_tokens_one_sequence_equals_repeated_single_appends():
    shape = tiny_shape(B=1, ctx=6, page_size=4)
    c1 = oc(tiny_cache(shape, num_pages=12, max_ctx=30))
    c2 = c1.copy()
    rng = np.random.default_rng(3)
    n = 11
    kb = rng.integers(0, 2**32, size=(1, n, shape.Hkv, shape.D), dtype=np.uint32)
    vb = rng.integers(0, 2**32, size=(1, n, shape.Hkv, shape.D), dtype=np.uint32)
    a1 = np.ones(c1.slot_map.shape)
    a2 = a1.copy()
    assert cache.append_tokens(c1, kb, vb, aux=a1) == cache.SE_OK
    for i in range(n):
        assert cache.append(c2, kb[:, i], vb[:, i], aux=a2) == cache.SE_OK
    for f in ("k", "v", "block_table", "slot_map", "ctx_len", "logical_len", "free_list",
              "page_refcount"):
        assert (getattr(c1, f) == getattr(c2, f)).all(), f
    assert c1.free_top == c2.free_top
    assert (a1 == a2).all()


def test_append_tokens_pop_order_and_contents():
    """Three sequences at ctx 22 (page 4) take 9 tokens each: blocks 6 and 7
    are fresh, popped from the stack top in (sequence, block) order."""
    shape = tiny_shape(B=3, ctx=22, page_size=4)
    c = oc(tiny_cache(shape, num_pages=48, max_ctx=32))
    before = c.copy()
    top = c.free_top
    rng = np.random.default_rng(5)
    kb = rng.integers(0, 2**32, size=(3, 9, shape.Hkv, shape.D), dtype=np.uint32)
    assert cache.append_tokens(c, kb, kb + 1) == cache.SE_OK
    assert c.free_top == top - 6
    stack = before.free_list
    for b in range(3):
        assert c.block_table[b, 6] == stack[top - 1 - 2 * b]
        assert c.block_table[b, 7] == stack[top - 2 - 2 * b]
        assert (c.block_table[b, :6] == before.block_table[b, :6]).all()
        for i in range(9):
            s = 22 + i
            assert (c.slot_map[b, :, s] == 22 + i).all()
            (p,), (r,) = c.where(b, [s])
            assert (c.k[p, :, r] == kb[b, i]).all() and (c.v[p, :, r] == kb[b, i] + 1).all()
    assert (c.ctx_len == 31).all() and (c.logical_len == 31).all()
    _check_accounting(before, c)


def test_append_tokens_errors_change_nothing():
    shape = tiny_shape(B=2, ctx=8, page_size=4)
    c = oc(tiny_cache(shape, num_pages=5, max_ctx=40))     # 4 pages used, 1 free
    before = c.copy()
    kb = np.zeros((2, 5, shape.Hkv, shape.D), dtype=np.uint32)
    assert cache.append_tokens(c, kb, kb) == cache.SE_ERR_OUT_OF_PAGES
    kb = np.zeros((2, 33, shape.Hkv, shape.D), dtype=np.uint32)
    assert cache.append_tokens(c, kb, kb) == cache.SE_ERR_BOUNDS
    for f in ("k", "block_table", "slot_map", "ctx_len", "free_list"):
        assert (getattr(c, f) == getattr(before, f)).all()
    assert c.free_top == before.free_top


def test_release_hand_worked_order_and_shared_page():
    """Sequences 0 and 2 of three (page 4) are released: pages go back in
    (sequence, block) order; a page held twice only loses a reference."""
    shape = tiny_shape(B=3, ctx=9, page_size=4)
    c = oc(tiny_cache(shape, num_pages=16, max_ctx=12))
    before = c.copy()
    shared = int(c.block_table[2, 1])
    c.page_refcount[shared] = 2                      # also held by someone else
    top = c.free_top
    assert cache.release(c, [1, 0, 1]) == cache.SE_OK
    expect = [int(p) for p in before.block_table[0, :3]] + \
        [int(before.block_table[2, 0]), int(before.block_table[2, 2])]
    assert list(c.free_list[top:c.free_top]) == expect
    assert c.page_refcount[shared] == 1 and shared not in c.free_list[:c.free_top]
    for b in (0, 2):
        assert (c.block_table[b] == -1).all() and (c.slot_map[b] == -1).all()
        assert c.ctx_len[b] == 0 and c.logical_len[b] == 0
    for f in ("block_table", "slot_map"):
        assert (getattr(c, f)[1] == getattr(before, f)[1]).all()
    assert c.ctx_len[1] == 9


@pytest.mark.parametrize("seed", range(3))
def test_release_conserves_pages(seed):
    rng = np.random.default_rng(seed)
    shape = tiny_shape(B=5, ctx=13, page_size=4)
    c = oc(tiny_cache(shape, num_pages=40, max_ctx=20))
    before = c.copy()
    mask = rng.integers(0, 2, size=5)
    assert cache.release(c, mask) == cache.SE_OK
    _check_accounting(before, c)
    released = sum(int((before.block_table[b] >= 0).sum()) for b in range(5) if mask[b])
    assert c.free_top == before.free_top + released


def test_kara_schedule_steps_untouched_and_compressed_sequences():
    """Staggered Kara compression in a decode loop: sequences whose window is
    not full only gain the appended token; a full window is cut to budget +
    protected entries (candidates kept, protected tail kept); attention output
    equals library SDPA over the resident entries before compression."""
    shape = W.kara_schedule(B=3, Hq=4, Hkv=2, D=16, ctx=40, window=16, protected=4,
                            candidates=4, budget=6, steps=14, dtype=torch.float32,
                            name="ks_tiny")
    inp = W.kara_schedule_inputs(shape, "cpu")
    c = oc(inp["cache"])
    ring = inp["q_ring"].clone()
    win_start = [shape.ctx - shape.fill(b) for b in range(3)]
    seen_due = 0
    for t in range(shape.steps):
        before = c.copy()
        r = pipelines.kara_schedule_step(c, inp["q_steps"][t], inp["k_steps"][t],
                                         inp["v_steps"][t], ring, win_start, shape)
        for b in range(3):
            n0 = int(before.ctx_len[b])
            if b in r["due"]:
                seen_due += 1
                lo = n0 + 1 - shape.window
                assert c.ctx_len[b] == lo + shape.budget + shape.protected
                for h in range(2):
                    kept = r["keep"][b][h]
                    assert len(kept) == shape.budget + shape.protected
                    assert set(range(n0 + 1 - shape.protected, n0 + 1)) <= set(kept.tolist())
            else:
                assert c.ctx_len[b] == n0 + 1
                assert (c.block_table[b, : before.block_table.shape[1]][before.block_table[b] >= 0]
                        == before.block_table[b][before.block_table[b] >= 0]).all()
            for g in range(2):
                Q = inp["q_steps"][t][b, g * shape.G:(g + 1) * shape.G].double().numpy()
                slots = np.arange(n0 + 1)
                # the appended entry is resident in the cache as it was after append
                cc = before.copy()
                cache.append(cc, cache._bits(inp["k_steps"][t]), cache._bits(inp["v_steps"][t]))
                ref = sdpa_out(Q, cc.keys(b, g, slots), cc.vals(b, g, slots))
                np.testing.assert_allclose(r["o"][(b, g)], ref, rtol=1e-12, atol=1e-13)
    assert seen_due >= 3


# ---------------------------------------------------------------------------
# O6 Quest
# ---------------------------------------------------------------------------


def _quest_tiny():
    shape = W.quest_decode(B=2, Hq=4, Hkv=2, D=16, ctx=64, page_size=4, top_pages=5, steps=2,
                           dtype=torch.bfloat16, name="quest_tiny")
    return shape, W.quest_inputs(shape, "cpu")


def test_quest_bound_is_upper_bound_and_meta_exact():
    shape, inp = _quest_tiny()
    c = oc(inp["cache"])
    kmin, kmax = quest.build_meta(c)
    q = values(cache._bits(inp["q_steps"][0]))
    for b in range(c.B):
        for blk in range(16):
            page = c.block_table[b, blk]
            for g in range(c.Hkv):
                K = c.keys(b, g, range(blk * 4, blk * 4 + 4))
                assert (kmin[page, g] <= K).all() and (K <= kmax[page, g]).all()
                assert ((K == kmin[page, g]).any(axis=0)).all() and ((K == kmax[page, g]).any(axis=0)).all()
                qg = q[b, g * 2:(g + 1) * 2]
                U = quest.page_bound(qg, kmin[page, g], kmax[page, g])
                for kv in K:
                    assert U >= float((qg @ kv).sum()) - 1e-12
                    for h in range(2):
                        assert quest.page_bound(qg[h:h + 1], kmin[page, g], kmax[page, g]) >= qg[h] @ kv - 1e-12


def test_quest_topk_brute_force_and_all_pages_dense():
    shape, inp = _quest_tiny()
    c = oc(inp["cache"])
    kmin, kmax = quest.build_meta(c)
    q = values(cache._bits(inp["q_steps"][1]))
    for b in range(c.B):
        for g in range(c.Hkv):
            sel, U = quest.select_pages(c, kmin, kmax, q, 5, b, g)
            ranked = sorted(range(15), key=lambda i: (-U[i], i))[:5]
            assert list(sel) == sorted(ranked) + [15]
    r = pipelines.quest_step(c, kmin, kmax, inp["q_steps"][1], 100)
    for (b, g), o in r["o"].items():
        slots = np.arange(64)
        qg = q[b, g * 2:(g + 1) * 2]
        np.testing.assert_allclose(o, sdpa_out(qg, c.keys(b, g, slots), c.vals(b, g, slots)),
                                   rtol=1e-12, atol=1e-14)


# ---------------------------------------------------------------------------
# O7 / O8 compaction, move-last, append, prune
# ---------------------------------------------------------------------------


def _hand_cache(P, block_table, ctx, free_stack, num_pages, D=2):
    B = len(block_table)
    maxp = max(len(r) for r in block_table)
    bt = np.full((B, maxp), -1, dtype=np.int64)
    for b, r in enumerate(block_table):
        bt[b, :len(r)] = r
    k = np.zeros((num_pages, 1, P, D), dtype=np.uint32)
    for p in range(num_pages):
        for r in range(P):
            k[p, 0, r, :] = 10 * p + r
    sm = np.full((B, 1, maxp * P), -1, dtype=np.int64)
    for b in range(B):
        sm[b, 0, :ctx[b]] = np.arange(ctx[b])
    fl = np.zeros(num_pages, dtype=np.int64)
    fl[:len(free_stack)] = free_stack
    refc = np.zeros(num_pages, dtype=np.int64)
    for r in block_table:
        for p in r:
            if p >= 0:
                refc[p] = 1
    return cache.Cache(k=k, v=k.copy(), block_table=bt, slot_map=sm,
                       ctx_len=np.array(ctx, dtype=np.int64), logical_len=np.array(ctx, dtype=np.int64),
                       free_list=fl, free_top=len(free_stack), page_refcount=refc, page_size=P)


def test_compact_golden_hand_example():
    g = golden("compact_freelist_hand.json")
    c = _hand_cache(g["page_size"], g["block_table"], g["ctx_len"], g["free_stack"], g["num_pages"])
    keep = [[np.array(x)] for x in g["keep"]]
    assert cache.compact(c, keep, g["first_slot"]) == cache.SE_OK
    e = g["expected"]
    assert c.block_table.tolist() == e["block_table"]
    assert c.ctx_len.tolist() == e["ctx_len"]
    assert c.free_list[: c.free_top].tolist() == e["free_stack"]
    assert c.slot_map[:, 0, :].tolist() == e["slot_map"]
    for page, rows in e["page_rows"].items():
        assert c.k[int(page), 0, :3, 0].tolist() == rows
    for page, rc in {**e["refcount_fresh"], **e["refcount_released"]}.items():
        assert c.page_refcount[int(page)] == rc


def _check_accounting(before, after):
    num = before.k.shape[0]
    in_tables = [int(p) for p in after.block_table.reshape(-1) if p >= 0]
    free = [int(p) for p in after.free_list[: after.free_top]]
    assert len(set(in_tables)) == len(in_tables)
    assert not set(in_tables) & set(free)
    assert sorted(in_tables + free) == list(range(num))


@pytest.mark.parametrize("seed", range(4))
def test_compact_conserves_entries_and_pages(seed):
    shape = tiny_shape(ctx=23, Hkv=3, Hq=6)
    pc = tiny_cache(shape, num_pages=40, tag=f"cc{seed}")
    c = oc(pc)
    before = c.copy()
    rng = np.random.default_rng(seed)
    first = [int(rng.integers(0, 23)) for _ in range(shape.B)]
    n_keep = [int(rng.integers(0, 23 - f + 1)) for f in first]
    keep = [[np.sort(rng.choice(np.arange(first[b], 23), n_keep[b], replace=False))
             for _ in range(3)] for b in range(shape.B)]
    assert cache.compact(c, keep, first) == cache.SE_OK
    _check_accounting(before, c)
    assert (c.logical_len == before.logical_len).all()
    for b in range(shape.B):
        assert c.ctx_len[b] == first[b] + n_keep[b]
        for h in range(3):
            old_pos = before.slot_map[b, h, :23]
            new_pos = c.slot_map[b, h, : c.ctx_len[b]]
            expect = list(old_pos[: first[b]]) + [old_pos[s] for s in keep[b][h]]
            assert list(new_pos) == expect
            evicted = sorted(set(old_pos.tolist()) - set(new_pos.tolist()))
            assert sorted(new_pos.tolist() + evicted) == sorted(old_pos.tolist())
            for i, s in enumerate(list(range(first[b])) + list(keep[b][h])):
                (p0,), (r0,) = before.where(b, [s])
                (p1,), (r1,) = c.where(b, [i])
                assert (before.k[p0, h, r0] == c.k[p1, h, r1]).all()
                assert (before.v[p0, h, r0] == c.v[p1, h, r1]).all()


def test_compact_out_of_pages_changes_nothing():
    shape = tiny_shape(ctx=20)
    c = oc(tiny_cache(shape, num_pages=10))
    c.free_top = 1
    before = c.copy()
    keep = [[np.arange(0, 10)] * 2 for _ in range(2)]
    assert cache.compact(c, keep, [0, 0]) == cache.SE_ERR_OUT_OF_PAGES
    assert (c.block_table == before.block_table).all() and c.free_top == 1


def test_compact_leaves_empty_rewrites_untouched():
    """Sequence 1 (ctx 21, not a page multiple) asks for an empty rewrite:
    nothing of it moves, while sequence 0 is compacted as usual."""
    shape = tiny_shape(B=2, ctx=21, page_size=4)
    c = oc(tiny_cache(shape, num_pages=30))
    before = c.copy()
    keep = [[np.array([9, 12, 20])] * 2, [np.array([], dtype=np.int64)] * 2]
    assert cache.compact(c, keep, [8, 21]) == cache.SE_OK
    assert (c.block_table[1] == before.block_table[1]).all()
    assert (c.slot_map[1] == before.slot_map[1]).all() and c.ctx_len[1] == 21
    assert c.ctx_len[0] == 11
    # only sequence 0's pages moved: one fresh page popped, its 4 old ones pushed
    assert c.free_top == before.free_top - 1 + 4
    _check_accounting(before, c)


def test_move_last_and_append():
    shape = tiny_shape(ctx=17, page_size=4)
    c = oc(tiny_cache(shape, num_pages=20, max_ctx=24))
    before = c.copy()
    victim = np.array([[3, 16], [0, 5]])
    assert cache.move_last(c, victim) == cache.SE_OK
    assert (c.ctx_len == 16).all()
    assert c.slot_map[0, 0, 3] == 16 and c.slot_map[0, 1, 16] == -1
    (p,), (r,) = before.where(0, [16])
    (q,), (s,) = c.where(0, [3])
    assert (c.k[q, 0, s] == before.k[p, 0, r]).all()
    assert c.free_top == before.free_top + 2          # block 4 emptied in both sequences
    _check_accounting(before, c)
    kb = np.full((2, 2, shape.D), 7, dtype=np.uint32)
    top = c.free_top
    assert cache.append(c, kb, kb) == cache.SE_OK
    assert c.free_top == top - 2 and (c.ctx_len == 17).all() and (c.logical_len == 18).all()
    assert c.slot_map[1, 1, 16] == 17
    _check_accounting(before, c)


def _prune_hand(busy):
    g = golden("prune_span_hand.json")
    c = _hand_cache(g["page_size"], [g["block_table"]], [g["ctx"]], g["free_stack"], 9)
    if busy:
        c.page_refcount[3] = 2
    st, nb = cache.prune(c, [g["L"]], [g["R"]], np.array([g["mask"]]))
    assert st == cache.SE_OK
    return g, c, nb


def test_prune_golden_hand_example_idle_and_busy():
    g, c, nb = _prune_hand(False)
    e = g["expected_idle"]
    assert c.slot_map[0, 0, : c.ctx_len[0]].tolist() == e["positions"]
    assert c.block_table[0].tolist() == e["block_table"]
    assert c.free_list[: c.free_top].tolist() == e["free_stack"]
    g, c, nb = _prune_hand(True)
    e = g["expected_busy"]
    assert c.slot_map[0, 0, : c.ctx_len[0]].tolist() == e["positions"]
    assert c.free_list[: c.free_top].tolist() == e["free_stack"]
    assert c.page_refcount[3] == e["refcount_page3"] and nb == [e["busy_pages"]]


@pytest.mark.parametrize("seed", range(4))
def test_prune_set_identity(seed):
    # Res' = (Res \ T) U I as Python sets, logical prefix unchanged
    shape = tiny_shape(ctx=40, page_size=4, Hkv=2)
    c = oc(tiny_cache(shape, num_pages=60, tag=f"pr{seed}"))
    rng = np.random.default_rng(seed)
    # first make head sets differ outside the span by an earlier compaction
    keep = [[np.sort(rng.choice(np.arange(30, 40), 6, replace=False)) for _ in range(2)]
            for _ in range(2)]
    assert cache.compact(c, keep, [30, 30]) == cache.SE_OK
    before = c.copy()
    L, R = [5, 9], [21, 30]
    mask = np.zeros((2, 25), dtype=np.uint8)
    for b in range(2):
        mask[b, rng.choice(R[b] - L[b], 4, replace=False)] = 1
    st, _ = cache.prune(c, L, R, mask)
    assert st == cache.SE_OK
    _check_accounting(before, c)
    assert (c.logical_len == before.logical_len).all()
    for b in range(2):
        T = set(range(L[b], R[b]))
        I = {L[b] + i for i in range(R[b] - L[b]) if mask[b, i]}
        for h in range(2):
            res = set(before.slot_map[b, h, : before.ctx_len[b]].tolist())
            new = c.slot_map[b, h, : c.ctx_len[b]].tolist()
            assert set(new) == (res - T) | (I & res)
            old_order = [p for p in before.slot_map[b, h, : before.ctx_len[b]].tolist() if p in set(new)]
            assert new == old_order


def test_prune_uneven_heads_is_rejected():
    shape = tiny_shape(ctx=16, page_size=4, Hkv=2)
    c = oc(tiny_cache(shape, num_pages=30))
    keep = [[np.array([0, 1, 2, 3, 4, 5]), np.array([0, 1, 2, 3, 10, 11])] for _ in range(2)]
    assert cache.compact(c, keep, [0, 0]) == cache.SE_OK
    mask = np.zeros((2, 4), dtype=np.uint8)
    st, _ = cache.prune(c, [2, 2], [6, 6], mask)
    assert st == cache.SE_ERR_UNEVEN


# ---------------------------------------------------------------------------
# O9 decode attention and the end-to-end full-budget identity
# ---------------------------------------------------------------------------


def test_decode_attention_matches_library_on_all_views():
    shape = tiny_shape(ctx=21, page_size=4)
    c = oc(tiny_cache(shape))
    q = torch.randn(2, shape.Hq, shape.D, generator=W.generator("cpu", "pin", "dq")).double().numpy()
    sel_p = {b: {g: np.array([0, 2, 5]) for g in range(2)} for b in range(2)}
    sel_t = {b: {g: np.array([1, 4, 9, 20]) for g in range(2)} for b in range(2)}
    for view, sel, slots in [("dense", None, np.arange(21)),
                             ("pages", sel_p, np.r_[0:4, 8:12, 20]),
                             ("tokens", sel_t, np.array([1, 4, 9, 20]))]:
        o, ps = attention.decode_attention(c, q, view, sel)
        for (b, g), ob in o.items():
            ref = sdpa_out(q[b, 2 * g:2 * g + 2], c.keys(b, g, slots), c.vals(b, g, slots))
            np.testing.assert_allclose(ob, ref, rtol=1e-12, atol=1e-14)
            assert ps[(b, g)][1].sum() == pytest.approx(2.0, rel=1e-12)


def test_decode_attention_special_cases():
    K = np.random.default_rng(0).standard_normal((1, 8))
    V = np.random.default_rng(1).standard_normal((1, 8))
    o, _ = attention.attend(np.ones((3, 8)), K, V)
    np.testing.assert_allclose(o, np.repeat(V, 3, 0))
    K = np.random.default_rng(2).standard_normal((9, 8))
    o, _ = attention.attend(np.ones((2, 8)), K, np.full((9, 8), 0.5))
    np.testing.assert_allclose(o, 0.5)


def test_snapkv_full_budget_reproduces_dense_attention():
    shape = W.snapkv_tiny(ctx=96, window=16, budget=96, heavy_count=3)
    inp = W.snapkv_inputs(shape, "cpu")
    c = oc(inp["cache"])
    before = c.copy()
    r = pipelines.snapkv(c, inp["q_win"], inp["q_pos"].numpy(), inp["q_dec"], shape)
    assert all(len(k) == 96 for kb in r["keep"] for k in kb)
    q = inp["q_dec"].double().numpy()
    for (b, g), o in r["o"].items():
        slots = np.arange(96)
        ref = sdpa_out(q[b, 4 * g:4 * g + 4], before.keys(b, g, slots), before.vals(b, g, slots))
        np.testing.assert_allclose(o, ref, rtol=1e-12, atol=1e-14)


def test_snapkv_tiny_workload_shape_facts():
    # the tiny SnapKV workload: budget 128 = top 96 + 32-token window, 8 fresh
    # pages taken, 32 old pages returned
    shape = W.snapkv_tiny()
    inp = W.snapkv_inputs(shape, "cpu")
    c = oc(inp["cache"])
    top0 = c.free_top
    r = pipelines.snapkv(c, inp["q_win"], inp["q_pos"].numpy(), inp["q_dec"], shape)
    keep = r["keep"][0][0]
    assert len(keep) == 128 and list(keep[-32:]) == list(range(480, 512))
    assert c.ctx_len[0] == 128 and c.free_top == top0 - 8 + 32
    assert (c.block_table[0, 8:] == -1).all()
