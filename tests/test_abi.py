"""The C-ABI library builds for sm_103a, loads, and exports every entry point
declared in include/se.h (no compute calls: this runs without a GPU)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    src = open(os.path.join(ROOT, "include", "se.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[\w]+\s*\*?\s*(se_\w+)\s*\(", src, flags=re.M)))


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    path = __graft_entry__._builder().build()
    return ctypes.CDLL(path)


def test_header_declares_the_six_path_calls():
    names = declared_functions()
    for n in ["se_score_window", "se_topk_select", "se_compact_evict", "se_prune_span",
              "se_quest_page_select", "se_sparse_decode_attn"]:
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert len(names) >= 14
    for n in names:
        assert hasattr(lib, n), n


def test_binding_covers_every_declared_symbol(lib):
    import attention_scored_sparse_gb300 as se
    assert sorted(se.EXPORTED) == declared_functions()


def test_status_strings_and_version(lib):
    import attention_scored_sparse_gb300 as se
    assert se.status_string(se.SE_ERR_OUT_OF_PAGES) == "SE_ERR_OUT_OF_PAGES"
    assert se.version() >= 100


def test_host_argument_errors_return_without_launch(lib):
    # a NULL descriptor and NULL tensors are caught on the host, before any launch
    import attention_scored_sparse_gb300 as se
    assert se._lib.se_score_window(None, None, 0, None, None, None, None, None, 0, 0, 0, None, 0,
                                   None, 0, None) == se.SE_ERR_INVALID_ARG
    kv = se.se_paged_kv()
    assert se._lib.se_compact_evict(ctypes.byref(kv), 0, None, 0, None, None, 0, None, 0, None, 0,
                                    None) == se.SE_ERR_INVALID_ARG


def test_struct_layout_matches_header():
    import attention_scored_sparse_gb300 as se
    assert ctypes.sizeof(se.se_paged_kv) == 10 * 8 + 8 * 4
    assert ctypes.sizeof(se.se_select_params) == 8 * 4
