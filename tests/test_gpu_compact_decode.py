"""se_compact_decode: compaction into fresh pages and decode attention over
the compacted cache in one pass over the kept entries (SparseEngine "How it
works": SnapKV's physical eviction after the last prompt chunk, then
attention through the AttentionView).

The cache must end bit for bit as the oracle's compaction leaves it, the
output must match the oracle's attention over the compacted cache, and on the
shapes where the one-pass kernel splits the work like decode attention does,
both must equal the two separate calls bit for bit.
"""
import numpy as np
import pytest
import torch

import se_workloads as W
from oracle import attention as oattn
from oracle import cache as ocache
from tests import gpu_helpers as H

pytestmark = pytest.mark.gpu


def _cache(dtype, D, G, *, B, Hkv, ctx, spare=40, tag):
    shape = W.Shape(name=tag, B=B, Hq=Hkv * G, Hkv=Hkv, D=D, page_size=16, ctx=ctx, dtype=dtype)
    pc = W.build_paged_cache(shape, num_pages=W.cdiv(ctx, 16) * B + spare, max_ctx=ctx,
                             device="cuda", tag=tag)
    q = W.normal((B, shape.Hq, D), dtype, "cuda", tag, "q")
    return shape, pc, q


def _args(keep, first, B, Hkv):
    width = max(max(len(k) for k in kb) for kb in keep)
    kt = H.keep_tensor(keep, B, Hkv, width, "cuda")
    n_keep = torch.tensor([len(keep[b][0]) for b in range(B)], dtype=torch.int32, device="cuda")
    fs = torch.tensor(first, dtype=torch.int32, device="cuda")
    return kt, n_keep, fs, max(width, 1)


def _fused(se, shape, pc, q, keep, first, max_entries, aux=None):
    kt, n_keep, fs, mk = _args(keep, first, shape.B, shape.Hkv)
    o = torch.full_like(q, float("nan"))
    se.se_compact_decode(se.kv_desc(pc, shape.Hq), kt, n_keep=n_keep, first_slot=fs, max_keep=mk,
                         q=q, o=o, max_entries=max_entries, aux=aux)
    return o


def _check_against_oracle(pc, c, shape, q, o):
    """c: the oracle cache after its compaction; o against attention over it."""
    H.assert_cache_equal(pc, c)
    oo, _ = oattn.decode_attention(c, q.double().cpu().numpy(), "dense")
    og = o.double().cpu().numpy()
    G = shape.G
    for (b, g), ref in oo.items():
        err = np.abs(og[b, g * G:(g + 1) * G] - ref).max()
        assert err <= H.OUT_ATOL[shape.dtype], (b, g, err)


@pytest.mark.parametrize("dtype,D,G", [(torch.bfloat16, 128, 4), (torch.bfloat16, 64, 2),
                                       (torch.float32, 128, 8), (torch.float32, 64, 4)])
@pytest.mark.parametrize("seed", [0, 1])
def test_compact_decode_matches_oracle(cuda_lib, dtype, D, G, seed):
    """Random first slots (an untouched prefix, a first rewritten page shared
    with it) and keep lists, running values moved with the entries."""
    se = cuda_lib
    shape, pc, q = _cache(dtype, D, G, B=3, Hkv=2, ctx=300, tag=f"cd{seed}{D}{G}")
    c = ocache.from_tensors(pc)
    keep, first = H.random_keep(c, 10 + seed)
    aux_np = np.random.default_rng(seed).random(c.slot_map.shape)
    aux = torch.from_numpy(aux_np.astype(np.float32)).cuda()
    aux_o = aux.double().cpu().numpy()
    assert ocache.compact(c, keep, first, aux=aux_o) == ocache.SE_OK
    o = _fused(se, shape, pc, q, keep, first, max_entries=300, aux=aux)
    torch.cuda.synchronize()
    assert H.status(pc) == 0
    _check_against_oracle(pc, c, shape, q, o)
    np.testing.assert_array_equal(aux.cpu().double().numpy(), aux_o)


def test_compact_decode_edge_sequences(cuda_lib):
    """Keep nothing, keep everything, a sequence left as it is (first slot at
    the context, nothing kept), two entries past a shared page."""
    se = cuda_lib
    shape, pc, q = _cache(torch.bfloat16, 128, 4, B=4, Hkv=2, ctx=37, tag="cdedge")
    c = ocache.from_tensors(pc)
    first = [0, 0, 37, 5]
    keep = [[np.array([], dtype=np.int64)] * 2, [np.arange(0, 37)] * 2,
            [np.array([], dtype=np.int64)] * 2, [np.array([5, 36])] * 2]
    assert ocache.compact(c, keep, first) == ocache.SE_OK
    o = _fused(se, shape, pc, q, keep, first, max_entries=37)
    torch.cuda.synchronize()
    assert H.status(pc) == 0
    H.assert_cache_equal(pc, c)
    og = o.double().cpu().numpy()
    assert (og[0] == 0).all()                     # nothing resident: zero output
    oo, _ = oattn.decode_attention(c, q.double().cpu().numpy(), "dense",
                                   groups=[(b, g) for b in (1, 2, 3) for g in range(2)])
    for (b, g), ref in oo.items():
        assert np.abs(og[b, g * 4:(g + 1) * 4] - ref).max() <= H.OUT_ATOL[torch.bfloat16]


def test_compact_decode_equals_separate_calls(cuda_lib):
    """SnapKV-shaped: 2 x 4 KV heads, 4096 tokens, 1024 kept per head (the
    last 64 forced).  Where the one-pass kernel splits each unit like decode
    attention does, cache and output equal se_compact_evict followed by
    se_sparse_decode_attn bit for bit."""
    se = cuda_lib
    B, Hkv, ctx, budget, win = 2, 4, 4096, 1024, 64
    outs = []
    for fused in (True, False):
        shape, pc, q = _cache(torch.bfloat16, 128, 4, B=B, Hkv=Hkv, ctx=ctx,
                              spare=B * W.cdiv(budget, 16) + 8, tag="cdsep")
        rng = np.random.default_rng(3)
        keep = [[np.concatenate([np.sort(rng.choice(ctx - win, budget - win, replace=False)),
                                 np.arange(ctx - win, ctx)]) for _ in range(Hkv)] for _ in range(B)]
        first = [0] * B
        if fused:
            o = _fused(se, shape, pc, q, keep, first, max_entries=budget)
        else:
            kt, n_keep, fs, mk = _args(keep, first, B, Hkv)
            kv = se.kv_desc(pc, shape.Hq)
            se.se_compact_evict(kv, se.SE_COMPACT_FRESH_PAGES, kt, n_keep=n_keep, first_slot=fs,
                                max_keep=mk)
            o = torch.empty_like(q)
            se.se_sparse_decode_attn(kv, q, view=se.SE_VIEW_DENSE, o=o, max_entries=budget)
        torch.cuda.synchronize()
        assert H.status(pc) == 0
        outs.append((pc, o))
    (pa, oa), (pb_, ob) = outs
    for name in ["block_table", "slot_map", "ctx_len", "free_list", "free_top", "page_refcount",
                 "k_pool", "v_pool"]:
        assert torch.equal(getattr(pa, name), getattr(pb_, name)), name
    assert torch.equal(oa, ob)


def test_compact_decode_long_view_runs_the_two_steps(cuda_lib):
    """10000 kept entries per (sequence, head): more than 16 CTAs of 512
    entries, so the call compacts and then attends in two steps, with the
    same results."""
    se = cuda_lib
    shape, pc, q = _cache(torch.bfloat16, 128, 4, B=1, Hkv=2, ctx=12000, spare=640, tag="cdlong")
    c = ocache.from_tensors(pc)
    keep, first = H.random_keep(c, 7, first=[0], frac=10000 / 12000)
    assert ocache.compact(c, keep, first) == ocache.SE_OK
    o = _fused(se, shape, pc, q, keep, first, max_entries=10000)
    torch.cuda.synchronize()
    assert H.status(pc) == 0
    _check_against_oracle(pc, c, shape, q, o)


@pytest.mark.parametrize("case", ["unsorted", "view_short", "out_of_pages"])
def test_compact_decode_refusals_leave_cache_unchanged(cuda_lib, case):
    """A keep list out of order, a compacted length beyond max_entries, or too
    few free pages: the status word says why and the cache does not move."""
    se = cuda_lib
    shape, pc, q = _cache(torch.bfloat16, 128, 4, B=3, Hkv=2, ctx=150, tag=f"cdref{case}")
    if case == "out_of_pages":
        pc.free_top.fill_(1)
    before = pc.clone()
    if case == "unsorted":
        keep, first, me, want = [[np.array([3, 2, 9])] * 2 for _ in range(3)], [0, 0, 0], 150, \
            se.SE_ERR_BOUNDS
    elif case == "view_short":
        keep, first, me, want = [[np.arange(10, 100)] * 2 for _ in range(3)], [0, 0, 0], 50, \
            se.SE_ERR_BOUNDS
    else:
        keep, first, me, want = [[np.arange(0, 140)] * 2 for _ in range(3)], [0, 0, 0], 150, \
            se.SE_ERR_OUT_OF_PAGES
    _fused(se, shape, pc, q, keep, first, max_entries=me)
    torch.cuda.synchronize()
    assert H.status(pc) == want
    for name in ["block_table", "slot_map", "ctx_len", "free_list", "free_top", "page_refcount"]:
        assert torch.equal(getattr(pc, name), getattr(before, name)), name


def test_compact_decode_reuses_its_workspace_after_a_refusal(cuda_lib):
    """Three calls on one workspace (one max_keep, so one size): a compaction,
    a refused one (a keep list out of order), and another compaction of the
    result.  Nothing of the refused call (its abort flag, its page counts)
    leaks into the next: the cache and output match the oracle after the
    third call."""
    se = cuda_lib
    B, Hkv, W_ = 3, 2, 300
    shape, pc, q = _cache(torch.bfloat16, 128, 4, B=B, Hkv=Hkv, ctx=300, spare=80, tag="cdws")
    kv = se.kv_desc(pc, shape.Hq)
    ws = torch.zeros(se._lib.se_compact_decode_workspace_size(kv, W_, 300), dtype=torch.uint8,
                     device="cuda")

    def call(keep, first, o):
        kt = H.keep_tensor(keep, B, Hkv, W_, "cuda")
        n_keep = torch.tensor([len(keep[b][0]) for b in range(B)], dtype=torch.int32, device="cuda")
        fs = torch.tensor(first, dtype=torch.int32, device="cuda")
        se.se_compact_decode(kv, kt, n_keep=n_keep, first_slot=fs, max_keep=W_, q=q, o=o,
                             max_entries=300, workspace=ws)
        torch.cuda.synchronize()

    c = ocache.from_tensors(pc)
    keep, first = H.random_keep(c, 21, first=[0, 40, 100], frac=0.6)
    assert ocache.compact(c, keep, first) == ocache.SE_OK
    call(keep, first, torch.empty_like(q))
    assert H.status(pc) == 0
    before = pc.clone()
    call([[np.array([5, 3])] * Hkv for _ in range(B)], [0] * B, torch.empty_like(q))
    assert H.status(pc) == se.SE_ERR_BOUNDS
    for name in ["block_table", "slot_map", "ctx_len", "free_list", "free_top", "page_refcount"]:
        assert torch.equal(getattr(pc, name), getattr(before, name)), name
    pc.status.zero_()
    keep2, first2 = H.random_keep(c, 22, frac=0.5)
    assert ocache.compact(c, keep2, first2) == ocache.SE_OK
    o2 = torch.full_like(q, float("nan"))
    call(keep2, first2, o2)
    assert H.status(pc) == 0
    _check_against_oracle(pc, c, shape, q, o2)
