"""GPU vs oracle: compaction, move-last eviction, append, prefix pruning.

Integer-exact work: block tables, slot maps, lengths, free list, reference
counts and every K/V byte of the touched sequences must match bit for bit.
Inputs (caches, keep lists, masks) come from the seeded generators only.
"""
import numpy as np
import pytest
import torch

import se_workloads as W
from oracle import cache as ocache
from tests import gpu_helpers as H

pytestmark = pytest.mark.gpu


def _cache(dtype, D, *, B=3, Hkv=2, ctx=150, P=16, spare=40, max_ctx=None, tag="c"):
    shape = W.Shape(name="cacheops", B=B, Hq=Hkv * 2, Hkv=Hkv, D=D, page_size=P, ctx=ctx, dtype=dtype)
    per = W.cdiv(max_ctx or ctx, P)
    pc = W.build_paged_cache(shape, num_pages=per * B + spare, max_ctx=max_ctx or ctx, device="cuda", tag=tag)
    return shape, pc


@pytest.mark.parametrize("dtype,D", [(torch.bfloat16, 128), (torch.bfloat16, 64),
                                     (torch.float32, 64), (torch.float32, 128)])
@pytest.mark.parametrize("seed", [0, 1, 2])
def test_compact_fresh_pages_matches_oracle(cuda_lib, dtype, D, seed):
    se = cuda_lib
    shape, pc = _cache(dtype, D, tag=f"cf{seed}")
    c = ocache.from_tensors(pc)
    keep, first = H.random_keep(c, seed)
    aux_np = np.random.default_rng(seed).random(c.slot_map.shape)
    aux = torch.from_numpy(aux_np.astype(np.float32)).cuda()
    aux_o = aux.double().cpu().numpy()
    assert ocache.compact(c, keep, first, aux=aux_o) == ocache.SE_OK
    width = max(len(keep[b][0]) for b in range(shape.B))
    kt = H.keep_tensor(keep, shape.B, shape.Hkv, width, "cuda")
    n_keep = torch.tensor([len(keep[b][0]) for b in range(shape.B)], dtype=torch.int32, device="cuda")
    fs = torch.tensor(first, dtype=torch.int32, device="cuda")
    se.se_compact_evict(se.kv_desc(pc, shape.Hq), se.SE_COMPACT_FRESH_PAGES, kt, n_keep=n_keep,
                        first_slot=fs, max_keep=max(width, 1), aux=aux)
    torch.cuda.synchronize()
    assert H.status(pc) == 0
    H.assert_cache_equal(pc, c)
    np.testing.assert_array_equal(aux.cpu().double().numpy(), aux_o)


def test_compact_edge_cases(cuda_lib):
    se = cuda_lib
    # keep nothing / keep everything / first slot at ctx, ragged page tails
    shape, pc = _cache(torch.bfloat16, 128, B=4, ctx=37, P=16, tag="edge")
    c = ocache.from_tensors(pc)
    first = [0, 0, 37, 5]
    keep = [[np.array([], dtype=np.int64)] * 2, [np.arange(0, 37)] * 2,
            [np.array([], dtype=np.int64)] * 2, [np.array([5, 36])] * 2]
    assert ocache.compact(c, keep, first) == ocache.SE_OK
    n_keep = torch.tensor([0, 37, 0, 2], dtype=torch.int32, device="cuda")
    kt = H.keep_tensor(keep, 4, 2, 37, "cuda")
    se.se_compact_evict(se.kv_desc(pc, shape.Hq), se.SE_COMPACT_FRESH_PAGES, kt, n_keep=n_keep,
                        first_slot=torch.tensor(first, dtype=torch.int32, device="cuda"), max_keep=37)
    torch.cuda.synchronize()
    assert H.status(pc) == 0
    H.assert_cache_equal(pc, c)


def test_compact_out_of_pages_leaves_cache_unchanged(cuda_lib):
    se = cuda_lib
    shape, pc = _cache(torch.bfloat16, 128, tag="oop")
    before = pc.clone()
    pc.free_top.fill_(1)
    c = ocache.from_tensors(pc)
    keep, first = H.random_keep(c, 5, first=[0, 0, 0], frac=0.9)
    kt = H.keep_tensor(keep, 3, 2, 150, "cuda")
    n_keep = torch.tensor([len(keep[b][0]) for b in range(3)], dtype=torch.int32, device="cuda")
    se.se_compact_evict(se.kv_desc(pc, shape.Hq), se.SE_COMPACT_FRESH_PAGES, kt, n_keep=n_keep,
                        first_slot=torch.zeros(3, dtype=torch.int32, device="cuda"), max_keep=150)
    torch.cuda.synchronize()
    assert H.status(pc) == se.SE_ERR_OUT_OF_PAGES
    for name in ["block_table", "slot_map", "ctx_len", "free_list", "page_refcount"]:
        assert torch.equal(getattr(pc, name), getattr(before, name)), name


def test_compact_rejects_unsorted_keep(cuda_lib):
    se = cuda_lib
    shape, pc = _cache(torch.bfloat16, 128, tag="uns")
    before = pc.clone()
    keep = [[np.array([3, 2, 9])] * 2 for _ in range(3)]
    kt = H.keep_tensor(keep, 3, 2, 3, "cuda")
    se.se_compact_evict(se.kv_desc(pc, shape.Hq), se.SE_COMPACT_FRESH_PAGES, kt,
                        n_keep=torch.full((3,), 3, dtype=torch.int32, device="cuda"),
                        first_slot=torch.zeros(3, dtype=torch.int32, device="cuda"), max_keep=3)
    torch.cuda.synchronize()
    assert H.status(pc) == se.SE_ERR_BOUNDS
    for name in ["block_table", "slot_map", "ctx_len", "free_list", "free_top"]:
        assert torch.equal(getattr(pc, name), getattr(before, name)), name


@pytest.mark.parametrize("ctx", [33, 48, 17])
def test_move_last_matches_oracle(cuda_lib, ctx):
    se = cuda_lib
    shape, pc = _cache(torch.bfloat16, 128, B=4, Hkv=3, ctx=ctx, tag=f"ml{ctx}")
    c = ocache.from_tensors(pc)
    rng = np.random.default_rng(ctx)
    victim = rng.integers(0, ctx, size=(4, 3))
    victim[1, :] = -1                     # sequence 1 evicts nothing
    victim[2, 0] = ctx - 1                # the last slot itself
    aux = torch.rand(c.slot_map.shape, generator=W.generator("cpu", "ml", ctx)).cuda()
    aux_o = aux.double().cpu().numpy()
    assert ocache.move_last(c, victim, aux=aux_o) == ocache.SE_OK
    se.se_compact_evict(se.kv_desc(pc, shape.Hq), se.SE_COMPACT_MOVE_LAST,
                        torch.from_numpy(victim.astype(np.int32)).cuda(), aux=aux)
    torch.cuda.synchronize()
    assert H.status(pc) == 0
    H.assert_cache_equal(pc, c)
    np.testing.assert_array_equal(aux.cpu().double().numpy(), aux_o)


def test_move_last_uneven_is_rejected(cuda_lib):
    se = cuda_lib
    shape, pc = _cache(torch.bfloat16, 128, B=2, Hkv=2, ctx=20, tag="mlu")
    before = pc.clone()
    victim = torch.tensor([[3, -1], [1, 2]], dtype=torch.int32, device="cuda")
    se.se_compact_evict(se.kv_desc(pc, shape.Hq), se.SE_COMPACT_MOVE_LAST, victim)
    torch.cuda.synchronize()
    assert H.status(pc) == se.SE_ERR_UNEVEN
    assert torch.equal(pc.ctx_len, before.ctx_len) and torch.equal(pc.slot_map, before.slot_map)


@pytest.mark.parametrize("dtype,D", [(torch.bfloat16, 128), (torch.float32, 64)])
def test_append_matches_oracle(cuda_lib, dtype, D):
    se = cuda_lib
    shape, pc = _cache(dtype, D, B=3, Hkv=2, ctx=31, max_ctx=40, tag="ap")
    c = ocache.from_tensors(pc)
    aux = torch.ones(c.slot_map.shape, device="cuda")
    aux_o = aux.double().cpu().numpy()
    for step in range(3):                 # crosses the page boundary at slot 32
        k = W.normal((3, 2, D), dtype, "cuda", "ap", "k", step)
        v = W.normal((3, 2, D), dtype, "cuda", "ap", "v", step)
        assert ocache.append(c, ocache._bits(k), ocache._bits(v), aux=aux_o) == ocache.SE_OK
        se.se_append_kv(se.kv_desc(pc, shape.Hq), k, v, aux=aux)
        torch.cuda.synchronize()
        assert H.status(pc) == 0
        H.assert_cache_equal(pc, c)
        np.testing.assert_array_equal(aux.cpu().double().numpy(), aux_o)


def test_append_keeps_quest_metadata_current(cuda_lib):
    # appending with kmin / kmax equals rebuilding the metadata from scratch
    se = cuda_lib
    from oracle import quest as oquest
    shape, pc = _cache(torch.bfloat16, 128, B=3, Hkv=2, ctx=29, max_ctx=60, tag="apq")
    kv = se.kv_desc(pc, shape.Hq)
    kmin = torch.empty_like(pc.k_pool[:, :, 0, :])
    kmax = torch.empty_like(kmin)
    se.se_quest_build_meta(kv, kmin, kmax)
    for step in range(20):                # crosses the page boundaries at 32 and 48
        k = W.normal((3, 2, 128), torch.bfloat16, "cuda", "apq", "k", step)
        se.se_append_kv(kv, k, k, kmin=kmin, kmax=kmax)
    torch.cuda.synchronize()
    assert H.status(pc) == 0
    c = ocache.from_tensors(pc)
    omin, omax = oquest.build_meta(c)
    for b in range(3):
        pages = c.block_table[b, : W.cdiv(int(c.ctx_len[b]), 16)]
        np.testing.assert_array_equal(kmin[pages].double().cpu().numpy(), omin[pages])
        np.testing.assert_array_equal(kmax[pages].double().cpu().numpy(), omax[pages])


@pytest.mark.parametrize("dtype,D,n", [(torch.bfloat16, 128, 37), (torch.float32, 64, 5),
                                         (torch.bfloat16, 128, 16)])
def test_append_chunk_matches_oracle(cuda_lib, dtype, D, n):
    """n tokens per sequence in one call (a prefill chunk), from a ragged
    start, with aux and Quest bounds kept current."""
    se = cuda_lib
    from oracle import quest as oquest
    shape, pc = _cache(dtype, D, B=3, Hkv=2, ctx=29, max_ctx=29 + 3 * n + 16, tag="apc")
    kv = se.kv_desc(pc, shape.Hq)
    c = ocache.from_tensors(pc)
    aux = torch.ones(c.slot_map.shape, device="cuda")
    aux_o = aux.double().cpu().numpy()
    kmin = torch.empty_like(pc.k_pool[:, :, 0, :])
    kmax = torch.empty_like(kmin)
    se.se_quest_build_meta(kv, kmin, kmax)
    for step in range(3):
        k = W.normal((3, n, 2, D), dtype, "cuda", "apc", "k", step)
        v = W.normal((3, n, 2, D), dtype, "cuda", "apc", "v", step)
        assert ocache.append_tokens(c, ocache._bits(k), ocache._bits(v), aux=aux_o) == ocache.SE_OK
        se.se_append_kv(kv, k, v, aux=aux, kmin=kmin, kmax=kmax)
        torch.cuda.synchronize()
        assert H.status(pc) == 0
        H.assert_cache_equal(pc, c)
        np.testing.assert_array_equal(aux.cpu().double().numpy(), aux_o)
    omin, omax = oquest.build_meta(c)
    for b in range(3):
        pages = c.block_table[b, : W.cdiv(int(c.ctx_len[b]), 16)]
        np.testing.assert_array_equal(kmin[pages].double().cpu().numpy(), omin[pages])
        np.testing.assert_array_equal(kmax[pages].double().cpu().numpy(), omax[pages])


def test_append_chunk_beyond_capacity_changes_nothing(cuda_lib):
    se = cuda_lib
    shape, pc = _cache(torch.bfloat16, 128, B=2, Hkv=2, ctx=20, max_ctx=48, tag="apb")
    before = pc.clone()
    k = W.normal((2, 29, 2, 128), torch.bfloat16, "cuda", "apb", "k")
    se.se_append_kv(se.kv_desc(pc, shape.Hq), k, k)
    torch.cuda.synchronize()
    assert H.status(pc) == se.SE_ERR_BOUNDS
    assert torch.equal(pc.ctx_len, before.ctx_len) and torch.equal(pc.block_table, before.block_table)
    assert torch.equal(pc.free_top, before.free_top)


@pytest.mark.parametrize("seed", range(3))
def test_release_matches_oracle(cuda_lib, seed):
    """Whole sequences give their pages back (a reclaimed chain's row): free
    list order, shared pages, cleared rows, bit for bit."""
    se = cuda_lib
    shape, pc = _cache(torch.bfloat16, 128, B=6, Hkv=2, ctx=70 + seed, max_ctx=96, tag=f"rel{seed}")
    rng = np.random.default_rng(seed)
    mask = rng.integers(0, 2, size=6).astype(np.int32)
    mask[seed % 6] = 1
    shared = int(pc.block_table[seed % 6, 1].item())
    pc.page_refcount[shared] = 2
    c = ocache.from_tensors(pc)
    assert ocache.release(c, mask) == ocache.SE_OK
    se.se_release_seqs(se.kv_desc(pc, shape.Hq), torch.tensor(mask, device="cuda"))
    torch.cuda.synchronize()
    assert H.status(pc) == 0
    H.assert_cache_equal(pc, c)
    np.testing.assert_array_equal(pc.page_refcount.cpu().numpy(), c.page_refcount)


def test_append_out_of_pages(cuda_lib):
    se = cuda_lib
    shape, pc = _cache(torch.bfloat16, 128, B=3, Hkv=2, ctx=32, max_ctx=48, tag="apo")
    pc.free_top.fill_(2)                  # three sequences need a page, two are free
    before = pc.clone()
    k = W.normal((3, 2, 128), torch.bfloat16, "cuda", "apo", "k")
    se.se_append_kv(se.kv_desc(pc, shape.Hq), k, k)
    torch.cuda.synchronize()
    assert H.status(pc) == se.SE_ERR_OUT_OF_PAGES
    assert torch.equal(pc.ctx_len, before.ctx_len) and torch.equal(pc.block_table, before.block_table)


def _gpu_compact(se, shape, pc, keep, first):
    width = max(max(len(k) for k in kb) for kb in keep)
    kt = H.keep_tensor(keep, shape.B, shape.Hkv, width, "cuda")
    n_keep = torch.tensor([len(keep[b][0]) for b in range(shape.B)], dtype=torch.int32, device="cuda")
    se.se_compact_evict(se.kv_desc(pc, shape.Hq), se.SE_COMPACT_FRESH_PAGES, kt, n_keep=n_keep,
                        first_slot=torch.tensor(first, dtype=torch.int32, device="cuda"),
                        max_keep=max(width, 1))


def test_compact_subset_leaves_other_sequences_untouched(cuda_lib):
    """One call compacts sequences 0 and 2; 1 and 3 (first slot = context,
    nothing kept) must not move at all."""
    se = cuda_lib
    shape, pc = _cache(torch.bfloat16, 128, B=4, Hkv=2, ctx=150, tag="sub")
    c = ocache.from_tensors(pc)
    rng = np.random.default_rng(4)
    keep, first = [], []
    for b in range(4):
        if b % 2 == 0:
            kb = np.sort(rng.choice(np.arange(40, 150), 37, replace=False))
            keep.append([kb, np.sort(rng.choice(np.arange(40, 150), 37, replace=False))])
            first.append(40)
        else:
            keep.append([np.array([], dtype=np.int64)] * 2)
            first.append(150)
    assert ocache.compact(c, keep, first) == ocache.SE_OK
    _gpu_compact(se, shape, pc, keep, first)
    torch.cuda.synchronize()
    assert H.status(pc) == 0
    H.assert_cache_equal(pc, c)


def _prune_case(se, seed, busy_pages=0):
    shape, pc = _cache(torch.bfloat16, 128, B=3, Hkv=2, ctx=200, spare=60, tag=f"pr{seed}")
    c = ocache.from_tensors(pc)
    # make head resident sets differ outside the span first: each side
    # compacts the tail with the same generated keep lists
    rng = np.random.default_rng(seed)
    keep = [[np.sort(rng.choice(np.arange(150, 200), 20, replace=False)) for _ in range(2)]
            for _ in range(3)]
    assert ocache.compact(c, keep, [150] * 3) == ocache.SE_OK
    _gpu_compact(se, shape, pc, keep, [150] * 3)
    torch.cuda.synchronize()
    H.assert_cache_equal(pc, c)
    for i in range(busy_pages):
        page = int(c.block_table[i % 3, 3 + i])
        c.page_refcount[page] = 2
        pc.page_refcount[page] = 2
    L, R = [20, 33, 5], [120, 101, 140]   # spans stay below the per-head tail at 150
    mask = np.zeros((3, 160), dtype=np.uint8)
    for b in range(3):
        mask[b, rng.choice(R[b] - L[b], (R[b] - L[b]) // 5, replace=False)] = 1
    return shape, pc, c, L, R, mask


@pytest.mark.parametrize("busy", [0, 2])
def test_prune_span_matches_oracle(cuda_lib, busy):
    se = cuda_lib
    shape, pc, c, L, R, mask = _prune_case(se, 7 + busy, busy)
    st, n_busy = ocache.prune(c, L, R, mask)
    assert st == ocache.SE_OK
    nb = torch.full((3,), -1, dtype=torch.int32, device="cuda")
    se.se_prune_span(se.kv_desc(pc, shape.Hq), torch.tensor(L, dtype=torch.int32, device="cuda"),
                     torch.tensor(R, dtype=torch.int32, device="cuda"),
                     torch.from_numpy(mask).cuda(), n_busy=nb)
    torch.cuda.synchronize()
    assert H.status(pc) == 0
    H.assert_cache_equal(pc, c)
    assert nb.cpu().tolist() == n_busy


def test_prune_span_long_context_matches_oracle(cuda_lib):
    """Contexts of several plan rounds (4601 slots; the plan scans 4096 a
    round) with a ragged tail, heads that differ above slot 4000 (each keeps
    its own 601 of the positions [4000, 5003)).  Sequence 0 prunes a span over
    both rounds; sequence 1's span starts where the heads differ, so the first
    rewritten slot is the lowest over the heads (everything in the span is kept,
    so the heads stay even); sequence 2's span lies past every position and
    leaves it as it is."""
    se = cuda_lib
    shape, pc = _cache(torch.bfloat16, 128, B=3, Hkv=2, ctx=5003, spare=300, tag="prl")
    c = ocache.from_tensors(pc)
    rng = np.random.default_rng(11)
    keep = [[np.sort(rng.choice(np.arange(4000, 5003), 601, replace=False)) for _ in range(2)]
            for _ in range(3)]
    assert ocache.compact(c, keep, [4000] * 3) == ocache.SE_OK
    _gpu_compact(se, shape, pc, keep, [4000] * 3)
    torch.cuda.synchronize()
    H.assert_cache_equal(pc, c)
    firsts = [int(np.argmax(c.slot_map[1, h, :4601] >= 4300)) for h in range(2)]
    assert firsts[0] != firsts[1]       # the heads reach the span at different slots
    L, R = [100, 4300, 6000], [3900, 5003, 7000]
    mask = np.zeros((3, 3800), dtype=np.uint8)
    mask[0, rng.choice(3800, 760, replace=False)] = 1
    mask[1, :] = 1
    st, n_busy = ocache.prune(c, L, R, mask)
    assert st == ocache.SE_OK
    nb = torch.full((3,), -1, dtype=torch.int32, device="cuda")
    se.se_prune_span(se.kv_desc(pc, shape.Hq), torch.tensor(L, dtype=torch.int32, device="cuda"),
                     torch.tensor(R, dtype=torch.int32, device="cuda"),
                     torch.from_numpy(mask).cuda(), n_busy=nb)
    torch.cuda.synchronize()
    assert H.status(pc) == 0
    H.assert_cache_equal(pc, c)
    assert nb.cpu().tolist() == n_busy
    assert int(c.ctx_len[2]) == 4601


def test_prune_uneven_heads_is_rejected(cuda_lib):
    se = cuda_lib
    shape, pc = _cache(torch.bfloat16, 128, B=1, Hkv=2, ctx=64, tag="pru")
    # head 0 keeps positions 0..31, head 1 keeps 0..15 and 40..55: a span over
    # [20, 40) holds 12 entries of head 0 and 0 of head 1
    keep = [[np.arange(0, 32), np.r_[0:16, 40:56]]]
    _gpu_compact(se, shape, pc, keep, [0])
    torch.cuda.synchronize()
    assert H.status(pc) == 0
    before = pc.clone()
    mask = torch.zeros((1, 20), dtype=torch.uint8, device="cuda")
    se.se_prune_span(se.kv_desc(pc, shape.Hq), torch.tensor([20], dtype=torch.int32, device="cuda"),
                     torch.tensor([40], dtype=torch.int32, device="cuda"), mask)
    torch.cuda.synchronize()
    assert H.status(pc) == se.SE_ERR_UNEVEN
    assert torch.equal(pc.slot_map, before.slot_map) and torch.equal(pc.ctx_len, before.ctx_len)
