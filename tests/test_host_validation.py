"""Host-side argument checks of the C ABI: every entry point rejects bad
shapes, modes and workspace sizes synchronously, before any launch (no GPU is
touched; the device pointers below are never dereferenced)."""
import ctypes

import pytest

import __graft_entry__

__graft_entry__._builder().build()
import attention_scored_sparse_gb300 as se  # noqa: E402

FAKE = ctypes.c_void_p(0x10000)   # non-null, never dereferenced on the host
L = se._lib


def kv(**kw):
    base = dict(B=2, Hq=8, Hkv=2, D=128, page_size=16, num_pages=64, max_pages_per_seq=8,
                dtype=se.SE_BF16)
    base.update(kw)
    d = se.se_paged_kv(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE,
                       base["B"], base["Hq"], base["Hkv"], base["D"], base["page_size"],
                       base["num_pages"], base["max_pages_per_seq"], base["dtype"])
    return ctypes.byref(d), d


@pytest.mark.parametrize("bad,code", [
    (dict(D=96), se.SE_ERR_UNSUPPORTED),
    (dict(page_size=12), se.SE_ERR_UNSUPPORTED),
    (dict(page_size=128), se.SE_ERR_UNSUPPORTED),
    (dict(dtype=7), se.SE_ERR_UNSUPPORTED),
    (dict(Hq=6, Hkv=4), se.SE_ERR_INVALID_ARG),
    (dict(B=0), se.SE_ERR_INVALID_ARG),
])
def test_descriptor_checks(bad, code):
    d, _ = kv(**bad)
    assert L.se_quest_build_meta(d, FAKE, FAKE, None) == code
    assert L.se_append_kv(d, FAKE, FAKE, 1, None, 0, None, None, FAKE, 1 << 20, None) == code


def test_null_pointers_rejected():
    d, raw = kv()
    raw.status = None
    assert L.se_quest_build_meta(ctypes.byref(raw), FAKE, FAKE, None) == se.SE_ERR_INVALID_ARG
    d, _ = kv()
    assert L.se_quest_build_meta(d, None, FAKE, None) == se.SE_ERR_INVALID_ARG


def test_score_window_workspace_and_sizes():
    d, _ = kv()
    need = L.se_score_window_workspace_size(d, 64, 4096)
    assert need > 0
    args = [d, FAKE, 64, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 0, 4096, FAKE, 4096, FAKE]
    assert L.se_score_window(*args, need - 1, None) == se.SE_ERR_INVALID_ARG
    bad_w = [d, FAKE, 0, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 0, 4096, FAKE, 4096, FAKE]
    assert L.se_score_window(*bad_w, need, None) == se.SE_ERR_INVALID_ARG
    assert L.se_score_window(d, None, 64, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 0, 4096, FAKE, 4096,
                             FAKE, need, None) == se.SE_ERR_INVALID_ARG


def test_topk_select_modes_and_parameters():
    d, _ = kv()

    def call(**kw):
        p = se.se_select_params(kw.get("mode", 0), kw.get("pool", 7), kw.get("k", 10),
                                kw.get("cb", 64), 0.01, kw.get("budget", 10), kw.get("recent", 4),
                                kw.get("n_max", 100))
        return L.se_topk_select(d, FAKE, 128, ctypes.byref(p), FAKE, FAKE, FAKE, FAKE, FAKE, 128,
                                FAKE, None)
    assert call(pool=6) == se.SE_ERR_INVALID_ARG          # even pooling kernel
    assert call(k=-1) == se.SE_ERR_INVALID_ARG
    assert call(mode=1, k=33) == se.SE_ERR_INVALID_ARG     # at most 32 Kara candidates
    assert call(mode=1, n_max=1000) == se.SE_ERR_UNSUPPORTED
    assert call(mode=2, budget=-1) == se.SE_ERR_INVALID_ARG
    assert call(mode=9) == se.SE_ERR_INVALID_ARG
    assert call(n_max=1 << 20) == se.SE_ERR_UNSUPPORTED    # beyond the radix kernels' range
    p = se.se_select_params(0, 1, 4, 0, 0.0, 0, 0, 10)
    # a forced range needs both ends
    assert L.se_topk_select(d, FAKE, 128, ctypes.byref(p), FAKE, FAKE, FAKE, None, FAKE, 128,
                            FAKE, None) == se.SE_ERR_INVALID_ARG


def test_compact_prune_decode_quest_argument_checks():
    d, _ = kv()
    ws = L.se_compact_evict_workspace_size(d, 100)
    # keep rows narrower than max_keep
    assert L.se_compact_evict(d, 0, FAKE, 50, FAKE, FAKE, 100, None, 0, FAKE, ws, None) == \
        se.SE_ERR_INVALID_ARG
    assert L.se_compact_evict(d, 0, FAKE, 100, FAKE, FAKE, 100, None, 0, FAKE, ws - 1, None) == \
        se.SE_ERR_INVALID_ARG
    assert L.se_compact_evict(d, 5, FAKE, 100, FAKE, FAKE, 100, None, 0, FAKE, ws, None) == \
        se.SE_ERR_INVALID_ARG
    pws = L.se_prune_span_workspace_size(d)
    assert L.se_prune_span(d, FAKE, FAKE, FAKE, 16, None, None, 0, FAKE, pws - 1, None) == \
        se.SE_ERR_INVALID_ARG
    dws = L.se_sparse_decode_attn_workspace_size(d, 128)
    assert L.se_sparse_decode_attn(d, FAKE, 1, None, 0, 4, 128, FAKE, None, 0, FAKE, dws, None) == \
        se.SE_ERR_INVALID_ARG                              # page view without a selection
    assert L.se_sparse_decode_attn(d, FAKE, 5, None, 0, 0, 128, FAKE, None, 0, FAKE, dws, None) == \
        se.SE_ERR_INVALID_ARG
    assert L.se_sparse_decode_attn(d, FAKE, 0, None, 0, 0, 128, FAKE, None, 0, FAKE, dws - 1, None) == \
        se.SE_ERR_INVALID_ARG
    qws = L.se_quest_page_select_workspace_size(d, 8)
    assert L.se_quest_page_select(d, FAKE, FAKE, FAKE, 4, 9, FAKE, None, FAKE, qws, None) == \
        se.SE_ERR_INVALID_ARG                              # more blocks than the table holds


def test_decode_rejects_pools_past_32_bit_row_indices():
    # K/V rows are indexed with 32-bit integers: a pool of 2^27 pages x 2 heads x 16
    # rows is refused on the host, before any launch
    d, _ = kv(num_pages=1 << 27)
    dws = 1 << 30
    assert L.se_sparse_decode_attn(d, FAKE, 0, None, 0, 0, 128, FAKE, None, 0, FAKE, dws, None) == \
        se.SE_ERR_UNSUPPORTED


def test_static_scratch_variant_checks_size_before_anything():
    d, _ = kv(B=64, Hkv=8, Hq=32)
    assert L.se_sparse_decode_attn_static(d, FAKE, 0, None, 0, 0, 1 << 22, FAKE, None, 0, None) == \
        se.SE_ERR_UNSUPPORTED
    assert L.se_sparse_decode_attn_static(d, FAKE, 0, None, 0, 0, 0, FAKE, None, 0, None) == \
        se.SE_ERR_INVALID_ARG


def test_append_meta_pointers_come_in_pairs():
    d, _ = kv()
    assert L.se_append_kv(d, FAKE, FAKE, 1, None, 0, FAKE, None, FAKE, 1 << 20, None) == \
        se.SE_ERR_INVALID_ARG


def test_append_token_count_checked_on_host():
    d, raw = kv()
    cap = raw.max_pages_per_seq * raw.page_size
    for n in (-1, cap + 1):
        assert L.se_append_kv(d, FAKE, FAKE, n, None, 0, None, None, FAKE, 1 << 20, None) == \
            se.SE_ERR_INVALID_ARG
    # zero tokens: nothing to launch
    assert L.se_append_kv(d, FAKE, FAKE, 0, None, 0, None, None, FAKE, 1 << 20, None) == se.SE_OK


def test_workspace_queries_grow_with_sizes():
    d, _ = kv()
    assert L.se_score_window_workspace_size(d, 64, 8192) >= L.se_score_window_workspace_size(d, 64, 4096)
    assert L.se_compact_evict_workspace_size(d, 512) >= L.se_compact_evict_workspace_size(d, 64)
    assert L.se_sparse_decode_attn_workspace_size(d, 4096) >= L.se_sparse_decode_attn_workspace_size(d, 128)


def test_quest_decode_step_host_checks():
    d, _ = kv()
    # null buffers, negative top
    assert L.se_quest_decode_step(d, None, FAKE, FAKE, 8, FAKE, None, None, None) == \
        se.SE_ERR_INVALID_ARG
    assert L.se_quest_decode_step(d, FAKE, FAKE, FAKE, -1, FAKE, None, None, None) == \
        se.SE_ERR_INVALID_ARG
    # more than 255 top pages, or a layout the fused kernel does not cover
    assert L.se_quest_decode_step(d, FAKE, FAKE, FAKE, 256, FAKE, None, None, None) == \
        se.SE_ERR_UNSUPPORTED
    d64, _ = kv(D=64)
    assert L.se_quest_decode_step(d64, FAKE, FAKE, FAKE, 8, FAKE, None, None, None) == \
        se.SE_ERR_UNSUPPORTED
    df, _ = kv(dtype=se.SE_F32)
    assert L.se_quest_decode_step(df, FAKE, FAKE, FAKE, 8, FAKE, None, None, None) == \
        se.SE_ERR_UNSUPPORTED


def test_release_seqs_host_checks():
    d, _ = kv()
    assert L.se_release_seqs(d, None, FAKE, 1 << 20, None) == se.SE_ERR_INVALID_ARG
    assert L.se_release_seqs(d, FAKE, None, 1 << 20, None) == se.SE_ERR_INVALID_ARG
    need = L.se_release_seqs_workspace_size(d)
    assert need > 0
    assert L.se_release_seqs(d, FAKE, FAKE, need - 1, None) == se.SE_ERR_INVALID_ARG
