"""se_score_window_one_launch: window scoring in one cooperative launch (bf16, D = 128, window rows of a
group within 256, key ranges of at least eight 128-key tiles): element-wise
parity with the oracle on ragged ranges, several waves, empty sequences,
repeated and accumulating calls on one workspace, and a bounded wait made to
run out (SparseEngine "How it works": SnapKV / H2O window scores; KARA
Method 1 for the bidirectional form).
"""
import numpy as np
import pytest
import torch

import se_workloads as W
from oracle import cache as ocache
from oracle import scoring as oscore
from tests import gpu_helpers as H

pytestmark = pytest.mark.gpu


def _case(tag, B, Hkv, G, w, ctx):
    shape = W.Shape(name=tag, B=B, Hq=Hkv * G, Hkv=Hkv, D=128, page_size=16, ctx=ctx,
                    dtype=torch.bfloat16)
    pc = W.build_paged_cache(shape, num_pages=B * W.cdiv(ctx, 16) + 3, max_ctx=ctx,
                             device="cuda", tag=tag)
    q_win = W.normal((B, w, shape.Hq, 128), torch.bfloat16, "cuda", tag, "q")
    return shape, pc, q_win


def _i32(x):
    return torch.tensor(x, dtype=torch.int32, device="cuda")


def _score(se, pc, shape, q_win, q_pos, lo, hi, olo, ohi, causal, n_max, scores, ws=None,
           accumulate=False):
    se.se_score_window_one_launch(se.kv_desc(pc, shape.Hq), q_win, q_pos, _i32(lo), _i32(hi), _i32(olo),
                       _i32(ohi), causal=causal, accumulate=accumulate, n_max=n_max,
                       scores=scores, workspace=ws)


def _check(pc, shape, q_win, q_pos, lo, hi, olo, ohi, causal, scores, fill):
    c = ocache.from_tensors(pc)
    ref = oscore.score_window(c, q_win, q_pos.cpu().numpy(), lo, hi, olo, ohi, causal)
    sg = scores.cpu().double().numpy()
    w = q_win.shape[1]
    for (b, g), row in ref.items():
        if len(row):
            H.assert_scores_close(sg[b, g, olo[b]:ohi[b]], row, torch.bfloat16, w, shape.G)
        assert (sg[b, g, :olo[b]] == fill).all() and (sg[b, g, ohi[b]:] == fill).all()


@pytest.mark.parametrize("causal", [True, False])
def test_fused_scores_ragged_ranges(cuda_lib, causal):
    """Four sequences: a page-misaligned range, a range ending inside a page,
    a window in the middle of the context, and an empty range."""
    se = cuda_lib
    B, Hkv, G, w, ctx = 4, 2, 4, 45, 3000
    shape, pc, q_win = _case("fused_rag", B, Hkv, G, w, ctx)
    q_pos = torch.arange(ctx - w, ctx, dtype=torch.int32).repeat(B, 1)
    q_pos[2] = torch.arange(1800, 1800 + w, dtype=torch.int32)
    q_pos = q_pos.cuda()
    lo, hi = [3, 0, 1100, 100], [3000, 2963, 2300, 100]
    olo, ohi = [10, 0, 1100, 100], [3000 - w, 2963, 2250, 100]
    scores = torch.full((B, Hkv, ctx + 4), -5.0, device="cuda")
    _score(se, pc, shape, q_win, q_pos, lo, hi, olo, ohi, causal, ctx, scores)
    torch.cuda.synchronize()
    assert H.status(pc) == 0
    _check(pc, shape, q_win, q_pos, lo, hi, olo, ohi, causal, scores, -5.0)


def test_fused_scores_several_waves(cuda_lib):
    """32 (sequence, KV head) groups of 8192 keys: the keys exceed one wave
    (three waves), and the wave boundaries fall between groups."""
    se = cuda_lib
    B, Hkv, G, w, ctx = 4, 8, 4, 64, 8192
    shape, pc, q_win = _case("fused_waves", B, Hkv, G, w, ctx)
    q_pos = torch.arange(ctx - w, ctx, dtype=torch.int32).repeat(B, 1).cuda()
    lo, hi, olo, ohi = [0] * B, [ctx] * B, [0] * B, [ctx - w] * B
    scores = torch.full((B, Hkv, ctx), -5.0, device="cuda")
    _score(se, pc, shape, q_win, q_pos, lo, hi, olo, ohi, True, ctx, scores)
    torch.cuda.synchronize()
    assert H.status(pc) == 0
    _check(pc, shape, q_win, q_pos, lo, hi, olo, ohi, True, scores, -5.0)


def test_fused_scores_repeat_and_accumulate(cuda_lib):
    """Calls on one workspace give the same scores bit for bit (the control
    block is left clean); an accumulating call adds the same scores."""
    se = cuda_lib
    B, Hkv, G, w, ctx = 2, 4, 4, 64, 2500
    shape, pc, q_win = _case("fused_rep", B, Hkv, G, w, ctx)
    q_pos = torch.arange(ctx - w, ctx, dtype=torch.int32).repeat(B, 1).cuda()
    lo, hi, olo, ohi = [0] * B, [ctx] * B, [0] * B, [ctx] * B
    ws = se.Workspace()
    runs = []
    for _ in range(2):
        s = torch.zeros((B, Hkv, ctx), device="cuda")
        _score(se, pc, shape, q_win, q_pos, lo, hi, olo, ohi, True, ctx, s, ws=ws)
        runs.append(s)
    acc = runs[0].clone()
    _score(se, pc, shape, q_win, q_pos, lo, hi, olo, ohi, True, ctx, acc, ws=ws, accumulate=True)
    torch.cuda.synchronize()
    assert H.status(pc) == 0
    assert torch.equal(runs[0], runs[1])
    torch.testing.assert_close(acc, 2 * runs[0], rtol=1e-6, atol=0)
    _check(pc, shape, q_win, q_pos, lo, hi, olo, ohi, True, runs[1], 0.0)


def test_fused_scores_wait_limit_runs_out(cuda_lib):
    """A wait limit of 1 ns in the workspace's control block: the first wait
    that is not already satisfied gives up, the status word reads
    SE_ERR_TIMEOUT and the launch winds down.  With the limit cleared and the
    status reset, the next call on the same workspace matches the oracle."""
    se = cuda_lib
    B, Hkv, G, w, ctx = 2, 4, 4, 64, 2500
    shape, pc, q_win = _case("fused_to", B, Hkv, G, w, ctx)
    q_pos = torch.arange(ctx - w, ctx, dtype=torch.int32).repeat(B, 1).cuda()
    lo, hi, olo, ohi = [0] * B, [ctx] * B, [0] * B, [ctx] * B
    kv = se.kv_desc(pc, shape.Hq)
    need = se._lib.se_score_window_workspace_size(kv, w, ctx)
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    limit = ws[:8].view(torch.int64)
    limit.fill_(1)
    scores = torch.zeros((B, Hkv, ctx), device="cuda")
    _score(se, pc, shape, q_win, q_pos, lo, hi, olo, ohi, True, ctx, scores, ws=ws)
    torch.cuda.synchronize()
    assert H.status(pc) == se.SE_ERR_TIMEOUT
    where = int(ws[12:16].view(torch.int32).item())
    assert where != 0                         # the first wait that gave up is recorded
    ws[12:16].zero_()
    limit.fill_(0)
    pc.status.zero_()
    scores.zero_()
    _score(se, pc, shape, q_win, q_pos, lo, hi, olo, ohi, True, ctx, scores, ws=ws)
    torch.cuda.synchronize()
    assert H.status(pc) == 0
    _check(pc, shape, q_win, q_pos, lo, hi, olo, ohi, True, scores, 0.0)
    # the tile counters and the count of finished CTAs are back at zero; the
    # call counter that tags merged rows has counted both calls
    assert int(ws[64:64 + 4 * B * Hkv].count_nonzero().item()) == 0
    assert int(ws[8:12].view(torch.int32).item()) == 0
    assert int(ws[16:20].view(torch.int32).item()) == 2


def test_fused_scores_equal_two_launch_scores(cuda_lib):
    """The one-launch form and the default form agree within the score
    tolerance on the Llama-shaped SnapKV window (4 x 8192 keys per group)."""
    se = cuda_lib
    B, Hkv, G, w, ctx = 4, 8, 4, 64, 8192
    shape, pc, q_win = _case("fused_vs", B, Hkv, G, w, ctx)
    q_pos = torch.arange(ctx - w, ctx, dtype=torch.int32).repeat(B, 1).cuda()
    lo, hi, olo, ohi = [0] * B, [ctx] * B, [0] * B, [ctx - w] * B
    s1 = torch.zeros((B, Hkv, ctx), device="cuda")
    s2 = torch.zeros_like(s1)
    _score(se, pc, shape, q_win, q_pos, lo, hi, olo, ohi, True, ctx, s1)
    se.se_score_window(se.kv_desc(pc, shape.Hq), q_win, q_pos, _i32(lo), _i32(hi), _i32(olo),
                       _i32(ohi), causal=True, accumulate=False, n_max=ctx, scores=s2)
    torch.cuda.synchronize()
    assert H.status(pc) == 0
    rel = ((s1 - s2).abs() / s2.abs().clamp_min(1e-12 * w * G)).max().item()
    assert rel <= 2e-3, rel


def test_fused_refuses_shapes_it_does_not_cover(cuda_lib):
    """Short key ranges (fewer than eight tiles) are refused without a launch."""
    se = cuda_lib
    shape, pc, q_win = _case("fused_no", 1, 1, 4, 8, 300)
    q_pos = torch.arange(292, 300, dtype=torch.int32)[None].cuda()
    scores = torch.full((1, 1, 300), -5.0, device="cuda")
    with pytest.raises(RuntimeError):
        _score(se, pc, shape, q_win, q_pos, [0], [300], [0], [300], True, 300, scores)
    torch.cuda.synchronize()
    assert (scores == -5.0).all()
