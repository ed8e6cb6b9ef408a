"""Allocation-free decode attention (se_sparse_decode_attn_static).

Some callers cannot allocate device memory where they call the library -- an
engine plugin that must not touch the allocator, a hook running while a
memory pool is locked, an embedded runtime with a fixed budget.  For them the
library offers one decode-attention entry point whose scratch lives in a
fixed 16 MiB device array the library itself defines.  This file checks,
through the C ABI, that two calls in a row -- and a third after an unrelated
call -- give the same outputs as the workspace-taking entry point, bit for
bit (the same kernels on the same inputs), and that a call needing more
scratch than the array holds is refused without a launch.  It is named so pytest collects it last.
"""
import ctypes

import pytest
import torch

import se_workloads as W

pytestmark = pytest.mark.gpu


def _case(tag):
    shape = W.Shape(name="noalloc", B=6, Hq=32, Hkv=8, D=128, page_size=16, ctx=1500,
                    dtype=torch.bfloat16)
    pc = W.build_paged_cache(shape, num_pages=6 * 94 + 2, max_ctx=1500, device="cuda", tag=tag)
    pc.ctx_len.copy_(torch.tensor([1500, 1499, 777, 16, 1, 1234], dtype=torch.int32))
    return shape, pc


def _static_call(se, kv, q, o, acc, max_entries, stream):
    rc = se._lib.se_sparse_decode_attn_static(
        ctypes.byref(kv), ctypes.c_void_p(q.data_ptr()), se.SE_VIEW_DENSE, None, 0, 0,
        max_entries, ctypes.c_void_p(o.data_ptr()),
        None if acc is None else ctypes.c_void_p(acc.data_ptr()),
        0 if acc is None else acc.shape[-1], stream)
    assert rc == se.SE_OK, se.status_string(rc)


def test_static_scratch_decode_matches_workspace_decode(cuda_lib):
    """Two calls in a row, then a third after an unrelated call has left other
    partial results in the shared array: each equals the workspace entry
    point's output and running scores bit for bit (same kernels, same split,
    same inputs), so nothing left in the array leaks into a result."""
    se = cuda_lib
    shape, pc = _case("noalloc")
    kv = se.kv_desc(pc, shape.Hq)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for call in range(3):
        if call == 2:
            # fill the array with partials of another batch (other keys,
            # queries and lengths)
            _, other = _case("noalloc_other")
            other.ctx_len.copy_(torch.tensor([1500, 3, 1500, 900, 1500, 64], dtype=torch.int32))
            kv_o = se.kv_desc(other, shape.Hq)
            q_o = W.normal((shape.B, shape.Hq, shape.D), shape.dtype, "cuda", "noalloc", "qo")
            _static_call(se, kv_o, q_o, torch.empty_like(q_o), None, 1500, stream)
        q = W.normal((shape.B, shape.Hq, shape.D), shape.dtype, "cuda", "noalloc", "q", call)
        acc_ref = torch.zeros((shape.B, shape.Hkv, 1504), device="cuda")
        acc = torch.zeros_like(acc_ref)
        o_ref = torch.empty_like(q)
        se.se_sparse_decode_attn(kv, q, view=se.SE_VIEW_DENSE, o=o_ref, max_entries=1500,
                                 acc_scores=acc_ref)
        o = torch.full_like(q, float("nan"))
        _static_call(se, kv, q, o, acc, 1500, stream)
        torch.cuda.synchronize()
        assert int(pc.status.item()) == 0
        assert torch.equal(o, o_ref), call
        assert torch.equal(acc, acc_ref), call


def test_static_scratch_refuses_oversized_calls(cuda_lib):
    se = cuda_lib
    shape, pc = _case("noalloc_big")
    kv = se.kv_desc(pc, shape.Hq)
    big = 1 << 22                              # needs far more than 16 MiB of scratch
    assert se._lib.se_sparse_decode_attn_workspace_size(ctypes.byref(kv), big) > \
        se.SE_DECODE_STATIC_SCRATCH_BYTES
    q = torch.zeros((shape.B, shape.Hq, shape.D), dtype=shape.dtype, device="cuda")
    o = torch.zeros_like(q)
    rc = se._lib.se_sparse_decode_attn_static(
        ctypes.byref(kv), ctypes.c_void_p(q.data_ptr()), se.SE_VIEW_DENSE, None, 0, 0, big,
        ctypes.c_void_p(o.data_ptr()), None, 0, None)
    assert rc == se.SE_ERR_UNSUPPORTED
