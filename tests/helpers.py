"""Small shared helpers for the tests (no method arithmetic here)."""
from __future__ import annotations

import numpy as np
import torch

import se_workloads as W


def tiny_shape(**kw) -> W.Shape:
    base = dict(name="tiny", B=2, Hq=4, Hkv=2, D=16, page_size=4, ctx=22, dtype=torch.float32)
    base.update(kw)
    return W.Shape(**base)


def tiny_cache(shape=None, *, num_pages=None, max_ctx=None, tag="t", device="cpu"):
    shape = shape or tiny_shape()
    per = W.cdiv(max_ctx or shape.ctx, shape.page_size)
    num_pages = num_pages or per * shape.B * 2 + 4
    return W.build_paged_cache(shape, num_pages=num_pages, max_ctx=max_ctx or shape.ctx,
                               device=device, tag=tag)


def sdpa_probs(Q: np.ndarray, K: np.ndarray, mask=None) -> np.ndarray:
    """Attention probabilities from torch's scaled_dot_product_attention with
    V = identity (library routine; fp64).  Q [m][D], K [n][D], mask [m][n]
    boolean (True = may attend)."""
    q = torch.from_numpy(Q)[None, None]
    k = torch.from_numpy(K)[None, None]
    v = torch.eye(K.shape[0], dtype=torch.float64)[None, None]
    am = None if mask is None else torch.from_numpy(np.asarray(mask))[None, None]
    return torch.nn.functional.scaled_dot_product_attention(q, k, v, attn_mask=am)[0, 0].numpy()


def sdpa_out(Q: np.ndarray, K: np.ndarray, V: np.ndarray) -> np.ndarray:
    q = torch.from_numpy(Q)[None, None]
    return torch.nn.functional.scaled_dot_product_attention(
        q, torch.from_numpy(K)[None, None], torch.from_numpy(V)[None, None])[0, 0].numpy()


def rel_err(a, b, floor=0.0):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return np.abs(a - b) / np.maximum(np.abs(b), floor)
