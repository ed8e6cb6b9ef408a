"""Python binding of the attention-scored sparse KV library (sm_103a, one GPU).

Argument marshalling only: every step runs in the CUDA kernels of
``_lib/libse_gb300.so`` (built from ``csrc/`` by ``build.py``); PyTorch only
provides device memory and streams.  The functions carry the C names of
``include/se.h``.  Importing the package fails when the library has not been
built -- there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os
from ctypes import POINTER, c_float, c_int32, c_int64, c_size_t, c_void_p

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libse_gb300.so")

SE_OK = 0
SE_ERR_INVALID_ARG = 1
SE_ERR_UNSUPPORTED = 2
SE_ERR_OUT_OF_PAGES = 3
SE_ERR_UNEVEN = 4
SE_ERR_BUSY = 5
SE_ERR_TIMEOUT = 6
SE_ERR_BOUNDS = 7
SE_ERR_CUDA = 8

SE_BF16, SE_F32 = 0, 1
SE_SELECT_TOPK, SE_SELECT_KARA_CHUNK, SE_SELECT_EVICT_ONE = 0, 1, 2
SE_COMPACT_FRESH_PAGES, SE_COMPACT_MOVE_LAST = 0, 1
SE_VIEW_DENSE, SE_VIEW_PAGES, SE_VIEW_TOKENS = 0, 1, 2
SE_DECODE_STATIC_SCRATCH_BYTES = 16 << 20

EXPORTED = [
    "se_score_window", "se_score_window_workspace_size", "se_score_window_one_launch",
    "se_topk_select",
    "se_compact_evict", "se_compact_evict_workspace_size",
    "se_compact_decode", "se_compact_decode_workspace_size",
    "se_prune_span", "se_prune_span_workspace_size",
    "se_quest_build_meta", "se_quest_page_select", "se_quest_page_select_workspace_size",
    "se_sparse_decode_attn", "se_sparse_decode_attn_workspace_size",
    "se_sparse_decode_attn_static",
    "se_append_kv", "se_append_kv_workspace_size", "se_quest_decode_step",
    "se_release_seqs", "se_release_seqs_workspace_size",
    "se_chain_index_create", "se_chain_index_destroy", "se_chain_acquire", "se_chain_finish",
    "se_chain_drop", "se_chain_count",
    "se_status_string", "se_version",
]


class se_paged_kv(ctypes.Structure):
    _fields_ = [
        ("k_pool", c_void_p), ("v_pool", c_void_p), ("block_table", c_void_p),
        ("slot_map", c_void_p), ("ctx_len", c_void_p), ("logical_len", c_void_p),
        ("free_list", c_void_p), ("free_top", c_void_p), ("page_refcount", c_void_p),
        ("status", c_void_p),
        ("B", c_int32), ("Hq", c_int32), ("Hkv", c_int32), ("D", c_int32),
        ("page_size", c_int32), ("num_pages", c_int32), ("max_pages_per_seq", c_int32),
        ("dtype", c_int32),
    ]


class se_select_params(ctypes.Structure):
    _fields_ = [
        ("mode", c_int32), ("pool_kernel", c_int32), ("k", c_int32),
        ("chunk_budget", c_int32), ("chunk_coef", c_float), ("budget", c_int32),
        ("recent", c_int32), ("n_max", c_int32),
    ]


class SEError(RuntimeError):
    def __init__(self, fn, code):
        super().__init__(f"{fn} returned {status_string(code)} ({code})")
        self.code = code


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    if not os.path.exists(path):
        raise ImportError(f"{path} is missing: build it with attention_scored_sparse_gb300.build")
    lib = ctypes.CDLL(path)
    P = POINTER(se_paged_kv)
    sigs = {
        "se_score_window": [P, c_void_p, c_int32, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                            c_int32, c_int32, c_int32, c_void_p, c_int64, c_void_p, c_size_t,
                            c_void_p],
        "se_score_window_one_launch": [P, c_void_p, c_int32, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                            c_int32, c_int32, c_int32, c_void_p, c_int64, c_void_p, c_size_t,
                            c_void_p],
        "se_score_window_workspace_size": [P, c_int32, c_int32],
        "se_topk_select": [P, c_void_p, c_int64, POINTER(se_select_params), c_void_p, c_void_p,
                           c_void_p, c_void_p, c_void_p, c_int32, c_void_p, c_void_p],
        "se_compact_evict": [P, c_int32, c_void_p, c_int32, c_void_p, c_void_p, c_int32, c_void_p,
                             c_int64, c_void_p, c_size_t, c_void_p],
        "se_compact_evict_workspace_size": [P, c_int32],
        "se_compact_decode": [P, c_void_p, c_int32, c_void_p, c_void_p, c_int32, c_void_p, c_int64,
                              c_void_p, c_void_p, c_int32, c_void_p, c_size_t, c_void_p],
        "se_compact_decode_workspace_size": [P, c_int32, c_int32],
        "se_prune_span": [P, c_void_p, c_void_p, c_void_p, c_int32, c_void_p, c_void_p, c_int64,
                          c_void_p, c_size_t, c_void_p],
        "se_prune_span_workspace_size": [P],
        "se_quest_build_meta": [P, c_void_p, c_void_p, c_void_p],
        "se_quest_page_select": [P, c_void_p, c_void_p, c_void_p, c_int32, c_int32, c_void_p,
                                 c_void_p, c_void_p, c_size_t, c_void_p],
        "se_quest_page_select_workspace_size": [P, c_int32],
        "se_sparse_decode_attn": [P, c_void_p, c_int32, c_void_p, c_int32, c_int32, c_int32,
                                  c_void_p, c_void_p, c_int64, c_void_p, c_size_t, c_void_p],
        "se_sparse_decode_attn_workspace_size": [P, c_int32],
        "se_sparse_decode_attn_static": [P, c_void_p, c_int32, c_void_p, c_int32, c_int32, c_int32,
                                         c_void_p, c_void_p, c_int64, c_void_p],
        "se_append_kv": [P, c_void_p, c_void_p, c_int32, c_void_p, c_int64, c_void_p, c_void_p,
                         c_void_p, c_size_t, c_void_p],
        "se_append_kv_workspace_size": [P],
        "se_quest_decode_step": [P, c_void_p, c_void_p, c_void_p, c_int32, c_void_p, c_void_p,
                                 c_void_p, c_void_p],
        "se_release_seqs": [P, c_void_p, c_void_p, c_size_t, c_void_p],
        "se_release_seqs_workspace_size": [P],
        "se_chain_index_create": [c_int32],
        "se_chain_index_destroy": [c_void_p],
        "se_chain_acquire": [c_void_p, c_void_p, c_int64, POINTER(c_int64), POINTER(c_int32),
                             POINTER(c_int64), POINTER(c_int32)],
        "se_chain_finish": [c_void_p, c_int64, c_void_p, c_int64],
        "se_chain_drop": [c_void_p, c_int64, POINTER(c_int32)],
        "se_chain_count": [c_void_p],
        "se_status_string": [c_int32],
        "se_version": [],
    }
    for name, args in sigs.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        if name.endswith("_workspace_size"):
            fn.restype = c_size_t
        elif name == "se_status_string":
            fn.restype = ctypes.c_char_p
        elif name == "se_chain_index_create":
            fn.restype = c_void_p
        elif name == "se_chain_index_destroy":
            fn.restype = None
        else:
            fn.restype = c_int32
    return lib


_lib = load_library()


def status_string(code: int) -> str:
    return _lib.se_status_string(int(code)).decode()


def version() -> int:
    return _lib.se_version()


# ---------------------------------------------------------------------------
# marshalling helpers
# ---------------------------------------------------------------------------


def _ptr(t):
    return None if t is None else c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _check(name, code):
    if code != SE_OK:
        raise SEError(name, code)


def kv_desc(cache, Hq: int) -> se_paged_kv:
    """Descriptor of a paged cache (an object with the tensors of
    ``se_workloads.PagedCache``)."""
    dt = {torch.bfloat16: SE_BF16, torch.float32: SE_F32}[cache.k_pool.dtype]
    num_pages, Hkv, P, D = cache.k_pool.shape
    return se_paged_kv(
        _ptr(cache.k_pool), _ptr(cache.v_pool), _ptr(cache.block_table), _ptr(cache.slot_map),
        _ptr(cache.ctx_len), _ptr(cache.logical_len), _ptr(cache.free_list), _ptr(cache.free_top),
        _ptr(getattr(cache, "page_refcount", None)), _ptr(cache.status),
        cache.block_table.shape[0], Hq, Hkv, D, P, num_pages, cache.block_table.shape[1], dt)


class Workspace:
    """Caller-owned scratch memory (a torch uint8 tensor, zeroed when
    allocated: the scoring call keeps a control block in it that must start
    at zero), grown on demand."""

    def __init__(self, device="cuda"):
        self.device = device
        self.buf = torch.empty(0, dtype=torch.uint8, device=device)

    def get(self, nbytes: int):
        if self.buf.numel() < nbytes:
            self.buf = torch.zeros(max(nbytes, 256), dtype=torch.uint8, device=self.device)
        return self.buf


def _ws(ws, nbytes, device):
    if ws is None:
        ws = torch.zeros(max(nbytes, 256), dtype=torch.uint8, device=device)
    elif isinstance(ws, Workspace):
        ws = ws.get(nbytes)
    if ws.numel() < nbytes:
        raise ValueError("workspace too small")
    return ws


# ---------------------------------------------------------------------------
# entry points (names of include/se.h)
# ---------------------------------------------------------------------------


def se_score_window(kv, q_win, q_pos, attn_lo, attn_hi, out_lo, out_hi, *, causal, accumulate,
                    n_max, scores, workspace=None, stream=None):
    d = ctypes.byref(kv)
    w = q_win.shape[1]
    need = _lib.se_score_window_workspace_size(d, w, n_max)
    ws = _ws(workspace, need, scores.device)
    _check("se_score_window", _lib.se_score_window(
        d, _ptr(q_win), w, _ptr(q_pos), _ptr(attn_lo), _ptr(attn_hi), _ptr(out_lo), _ptr(out_hi),
        int(causal), int(accumulate), n_max, _ptr(scores), scores.shape[-1], _ptr(ws), ws.numel(),
        _stream(stream)))


def se_score_window_one_launch(kv, q_win, q_pos, attn_lo, attn_hi, out_lo, out_hi, *, causal,
                               accumulate, n_max, scores, workspace=None, stream=None):
    """se_score_window with both sweeps in one cooperative launch (see se.h)."""
    d = ctypes.byref(kv)
    w = q_win.shape[1]
    need = _lib.se_score_window_workspace_size(d, w, n_max)
    ws = _ws(workspace, need, scores.device)
    _check("se_score_window_one_launch", _lib.se_score_window_one_launch(
        d, _ptr(q_win), w, _ptr(q_pos), _ptr(attn_lo), _ptr(attn_hi), _ptr(out_lo), _ptr(out_hi),
        int(causal), int(accumulate), n_max, _ptr(scores), scores.shape[-1], _ptr(ws), ws.numel(),
        _stream(stream)))


def se_topk_select(kv, scores, *, mode, cand_lo=None, cand_hi=None, force_lo=None, force_hi=None,
                   keep_idx, n_keep=None, pool_kernel=1, k=0, chunk_budget=0, chunk_coef=0.0,
                   budget=0, recent=0, n_max=0, stream=None):
    p = se_select_params(mode, pool_kernel, k, chunk_budget, chunk_coef, budget, recent, n_max)
    keep_stride = keep_idx.shape[-1] if keep_idx.dim() == 3 else 1
    _check("se_topk_select", _lib.se_topk_select(
        ctypes.byref(kv), _ptr(scores), scores.shape[-1], ctypes.byref(p), _ptr(cand_lo),
        _ptr(cand_hi), _ptr(force_lo), _ptr(force_hi), _ptr(keep_idx), keep_stride, _ptr(n_keep),
        _stream(stream)))


def se_compact_evict(kv, mode, keep_idx, *, n_keep=None, first_slot=None, max_keep=0, aux=None,
                     workspace=None, stream=None):
    d = ctypes.byref(kv)
    need = _lib.se_compact_evict_workspace_size(d, max_keep)
    ws = _ws(workspace, need, keep_idx.device)
    keep_stride = keep_idx.shape[-1] if keep_idx.dim() == 3 else 1
    _check("se_compact_evict", _lib.se_compact_evict(
        d, mode, _ptr(keep_idx), keep_stride, _ptr(n_keep), _ptr(first_slot), max_keep, _ptr(aux),
        aux.shape[-1] if aux is not None else 0, _ptr(ws), ws.numel(), _stream(stream)))


def se_compact_decode(kv, keep_idx, *, n_keep, first_slot, max_keep, q, o, max_entries,
                      aux=None, workspace=None, stream=None):
    d = ctypes.byref(kv)
    need = _lib.se_compact_decode_workspace_size(d, max_keep, max_entries)
    ws = _ws(workspace, need, keep_idx.device)
    _check("se_compact_decode", _lib.se_compact_decode(
        d, _ptr(keep_idx), keep_idx.shape[-1], _ptr(n_keep), _ptr(first_slot), max_keep, _ptr(aux),
        aux.shape[-1] if aux is not None else 0, _ptr(q), _ptr(o), max_entries, _ptr(ws),
        ws.numel(), _stream(stream)))


def se_prune_span(kv, L, R, mask, *, n_busy=None, aux=None, workspace=None, stream=None):
    d = ctypes.byref(kv)
    need = _lib.se_prune_span_workspace_size(d)
    ws = _ws(workspace, need, mask.device)
    _check("se_prune_span", _lib.se_prune_span(
        d, _ptr(L), _ptr(R), _ptr(mask), mask.shape[-1], _ptr(n_busy), _ptr(aux),
        aux.shape[-1] if aux is not None else 0, _ptr(ws), ws.numel(), _stream(stream)))


def se_quest_build_meta(kv, kmin, kmax, stream=None):
    _check("se_quest_build_meta", _lib.se_quest_build_meta(
        ctypes.byref(kv), _ptr(kmin), _ptr(kmax), _stream(stream)))


def se_quest_page_select(kv, kmin, kmax, q, *, top_pages, max_blocks, page_idx, n_sel=None,
                         workspace=None, stream=None):
    d = ctypes.byref(kv)
    need = _lib.se_quest_page_select_workspace_size(d, max_blocks)
    ws = _ws(workspace, need, q.device)
    _check("se_quest_page_select", _lib.se_quest_page_select(
        d, _ptr(kmin), _ptr(kmax), _ptr(q), top_pages, max_blocks, _ptr(page_idx), _ptr(n_sel),
        _ptr(ws), ws.numel(), _stream(stream)))


def se_sparse_decode_attn(kv, q, *, view, o, max_entries, sel=None, n_sel=0, acc_scores=None,
                          workspace=None, stream=None):
    d = ctypes.byref(kv)
    need = _lib.se_sparse_decode_attn_workspace_size(d, max_entries)
    ws = _ws(workspace, need, q.device)
    sel_stride = sel.shape[-1] if sel is not None else 0
    _check("se_sparse_decode_attn", _lib.se_sparse_decode_attn(
        d, _ptr(q), view, _ptr(sel), sel_stride, n_sel, max_entries, _ptr(o), _ptr(acc_scores),
        acc_scores.shape[-1] if acc_scores is not None else 0, _ptr(ws), ws.numel(),
        _stream(stream)))


def se_sparse_decode_attn_static(kv, q, *, view, o, max_entries, sel=None, n_sel=0,
                                 acc_scores=None, stream=None):
    """Decode attention with the library's fixed device scratch (no workspace)."""
    sel_stride = sel.shape[-1] if sel is not None else 0
    _check("se_sparse_decode_attn_static", _lib.se_sparse_decode_attn_static(
        ctypes.byref(kv), _ptr(q), view, _ptr(sel), sel_stride, n_sel, max_entries, _ptr(o),
        _ptr(acc_scores), acc_scores.shape[-1] if acc_scores is not None else 0,
        _stream(stream)))


def se_append_kv(kv, k_new, v_new, *, aux=None, kmin=None, kmax=None, workspace=None,
                 stream=None):
    """k_new, v_new: [B][Hkv][D] (one token per sequence) or [B][n][Hkv][D]."""
    d = ctypes.byref(kv)
    n_new = 1 if k_new.dim() == 3 else k_new.shape[1]
    need = _lib.se_append_kv_workspace_size(d)
    ws = _ws(workspace, need, k_new.device)
    _check("se_append_kv", _lib.se_append_kv(
        d, _ptr(k_new), _ptr(v_new), n_new, _ptr(aux), aux.shape[-1] if aux is not None else 0,
        _ptr(kmin), _ptr(kmax), _ptr(ws), ws.numel(), _stream(stream)))


def se_quest_decode_step(kv, kmin, kmax, q, o, *, top_pages, page_idx=None, n_sel=None,
                         stream=None):
    _check("se_quest_decode_step", _lib.se_quest_decode_step(
        ctypes.byref(kv), _ptr(kmin), _ptr(kmax), _ptr(q), top_pages, _ptr(o), _ptr(page_idx),
        _ptr(n_sel), _stream(stream)))


def se_release_seqs(kv, mask, *, workspace=None, stream=None):
    """mask: device int32 [B]; 1 = give back every page of that sequence."""
    d = ctypes.byref(kv)
    need = _lib.se_release_seqs_workspace_size(d)
    ws = _ws(workspace, need, mask.device)
    _check("se_release_seqs", _lib.se_release_seqs(d, _ptr(mask), _ptr(ws), ws.numel(),
                                                   _stream(stream)))


class ChainIndex:
    """Host-side chain index (see se_chain_acquire in se.h): which cache row
    holds which session, matched on logical token prefixes, idle chains
    reclaimed least recently used first."""

    def __init__(self, n_rows: int):
        self._h = _lib.se_chain_index_create(n_rows)
        if not self._h:
            raise ValueError("could not create a chain index")

    def close(self):
        if self._h:
            _lib.se_chain_index_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    @staticmethod
    def _tokens(tokens):
        arr = (ctypes.c_int32 * max(len(tokens), 1))(*[int(t) for t in tokens])
        return arr, len(tokens)

    def acquire(self, tokens):
        """Returns (chain_id, row, reuse_len, reclaimed_row); SEError BUSY when
        every row serves a request."""
        arr, n = self._tokens(tokens)
        cid, row, reuse, rec = c_int64(), c_int32(), c_int64(), c_int32()
        _check("se_chain_acquire", _lib.se_chain_acquire(
            self._h, ctypes.cast(arr, c_void_p), n, ctypes.byref(cid), ctypes.byref(row),
            ctypes.byref(reuse), ctypes.byref(rec)))
        return cid.value, row.value, reuse.value, rec.value

    def finish(self, chain_id, tokens):
        arr, n = self._tokens(tokens)
        _check("se_chain_finish", _lib.se_chain_finish(self._h, chain_id,
                                                       ctypes.cast(arr, c_void_p), n))

    def drop(self, chain_id) -> int:
        row = c_int32()
        _check("se_chain_drop", _lib.se_chain_drop(self._h, chain_id, ctypes.byref(row)))
        return row.value

    def __len__(self):
        return _lib.se_chain_count(self._h)


def workspace_sizes(kv, *, w=1, n_max=1, max_keep=0, max_blocks=1, max_entries=1) -> dict:
    d = ctypes.byref(kv)
    return {
        "score_window": _lib.se_score_window_workspace_size(d, w, n_max),
        "compact_evict": _lib.se_compact_evict_workspace_size(d, max_keep),
        "compact_decode": _lib.se_compact_decode_workspace_size(d, max_keep, max_entries),
        "prune_span": _lib.se_prune_span_workspace_size(d),
        "quest_page_select": _lib.se_quest_page_select_workspace_size(d, max_blocks),
        "sparse_decode_attn": _lib.se_sparse_decode_attn_workspace_size(d, max_entries),
        "append_kv": _lib.se_append_kv_workspace_size(d),
        "release_seqs": _lib.se_release_seqs_workspace_size(d),
    }
