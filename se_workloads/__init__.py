"""Seeded synthetic inputs shaped like the five attention-scored sparse KV workloads.

This module only draws random numbers and lays them out in the paged-cache
format that both the CUDA library and the CPU oracle read.  It holds none of the
method's arithmetic (no scoring, selection, compaction or attention): the
oracle under ``oracle/`` and the CUDA path under ``attention_scored_sparse_gb300/``
both receive the tensors built here and nothing else.

Generation recipe (same for every workload):

* values are drawn N(0, 1) in fp32 by a seeded ``torch.Generator`` on the
  target device and rounded to nearest-even into the workload dtype (bf16 or
  fp32); the oracle reads the very same tensors, widened exactly to fp64;
* physical pages are handed out by a seeded permutation of the page pool, so
  block tables are scattered the way a long-running paged cache is; pages
  not handed out form the free list (a stack, top at the end);
* "heavy" keys follow the workload text: the tiny SnapKV case scales the
  whole key vector by 4 at 8 seeded positions of the scored prefix; the
  Llama-3.1-8B-shaped SnapKV case adds 3*u (u a seeded unit vector per
  sequence and KV head) at floor(1% of the scored prefix) seeded positions;
* the prune mask keeps exactly floor(0.2 * span) positions of [L, R), drawn
  without replacement and shared by all KV heads of a sequence.

Each tensor has its own generator stream: seed = hash of (base seed,
workload name, tensor name).
"""
from __future__ import annotations

import dataclasses
import hashlib
import math
from typing import Optional

import torch

BASE_SEED = 20261202


def stream_seed(*parts) -> int:
    """Deterministic 63-bit seed for one named tensor stream."""
    h = hashlib.sha256(("/".join(str(p) for p in (BASE_SEED,) + parts)).encode()).digest()
    return int.from_bytes(h[:8], "little") & ((1 << 63) - 1)


def generator(device, *parts) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(stream_seed(*parts))
    return g


def normal(shape, dtype, device, *parts) -> torch.Tensor:
    """N(0,1) drawn in fp32, rounded to nearest-even into ``dtype``."""
    g = generator(device, *parts)
    x = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    return x.to(dtype)


def choose(n: int, k: int, *parts) -> torch.Tensor:
    """k distinct indices of range(n), seeded, sorted ascending (host, int64)."""
    g = generator("cpu", *parts)
    return torch.sort(torch.randperm(n, generator=g)[:k]).values


# ----------------------------------------------------------------------------
# Workload shapes
# ----------------------------------------------------------------------------


@dataclasses.dataclass
class Shape:
    name: str
    B: int
    Hq: int
    Hkv: int
    D: int
    page_size: int
    ctx: int              # resident tokens per sequence when the workload starts
    dtype: torch.dtype

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv


@dataclasses.dataclass
class SnapKV(Shape):
    """End-of-prefill SnapKV compression: window scoring, pooling, top-k, compaction."""
    window: int = 32
    pool_kernel: int = 7
    budget: int = 128          # includes the window
    heavy_count: int = 8
    heavy_mode: str = "scale4"  # "scale4" (tiny case) or "offset3u" (Llama-shaped)

    @property
    def scored(self) -> int:
        return self.ctx - self.window

    @property
    def keep_topk(self) -> int:
        return self.budget - self.window


@dataclasses.dataclass
class Quest(Shape):
    """Query-dependent page selection over per-page key min/max, then sparse decode."""
    top_pages: int = 128
    steps: int = 64


@dataclasses.dataclass
class H2O(Shape):
    """Accumulated-score eviction: prompt compression, then decode with evict-one."""
    heavy: int = 1024
    recent: int = 128
    steps: int = 512

    @property
    def budget(self) -> int:
        return self.heavy + self.recent


@dataclasses.dataclass
class Kara(Shape):
    """Sliding-window bidirectional scoring + Token2Chunk, then prefix-span pruning."""
    window: int = 256
    protected: int = 32
    candidates: int = 32
    budget: int = 64
    chunk_coef: float = 0.01
    prune_L: int = 2048
    prune_R: int = 6144
    prune_keep_frac: float = 0.2

    @property
    def compressible(self) -> int:
        return self.window - self.protected

    @property
    def prune_keep(self) -> int:
        return int(math.floor(self.prune_keep_frac * (self.prune_R - self.prune_L)))


@dataclasses.dataclass
class KaraSchedule(Kara):
    """Kara compression inside a decode loop, staggered across the batch:
    every sequence compresses its trailing window whenever it fills, and the
    sequences start at different fills so that only a few compress per step."""
    steps: int = 320

    @property
    def period(self) -> int:
        """Decode steps between two compressions of one sequence."""
        return self.window - (self.budget + self.protected)

    def fill(self, b: int) -> int:
        """Window fill of sequence b before the first step."""
        return self.budget + self.protected + (b * self.period // self.B) % self.period


def snapkv_tiny(**kw) -> SnapKV:
    """1 sequence, GQA 4 (4 query heads / 1 KV head), d=64, fp32, 512 tokens."""
    base = dict(name="snapkv_tiny", B=1, Hq=4, Hkv=1, D=64, page_size=16, ctx=512,
                dtype=torch.float32, window=32, pool_kernel=7, budget=128,
                heavy_count=8, heavy_mode="scale4")
    base.update(kw)
    return SnapKV(**base)


def snapkv_llama8b(**kw) -> SnapKV:
    """Llama-3.1-8B-shaped layer: 4 x 32768 tokens, 32/8 heads, d=128, bf16."""
    base = dict(name="snapkv_llama8b", B=4, Hq=32, Hkv=8, D=128, page_size=16, ctx=32768,
                dtype=torch.bfloat16, window=64, pool_kernel=7, budget=2048,
                heavy_count=-1, heavy_mode="offset3u")
    base.update(kw)
    return SnapKV(**base)


def quest_decode(**kw) -> Quest:
    """2 x 131072 tokens, 32/8 heads, d=128, bf16, top 128 pages + current."""
    base = dict(name="quest_decode", B=2, Hq=32, Hkv=8, D=128, page_size=16, ctx=131072,
                dtype=torch.bfloat16, top_pages=128, steps=64)
    base.update(kw)
    return Quest(**base)


def h2o_decode(**kw) -> H2O:
    """Qwen3-4B-like layer: 64 sequences, 4096-token prompt, 1024+128 budget, 512 steps."""
    base = dict(name="h2o_decode", B=64, Hq=32, Hkv=8, D=128, page_size=16, ctx=4096,
                dtype=torch.bfloat16, heavy=1024, recent=128, steps=512)
    base.update(kw)
    return H2O(**base)


def kara_prune(**kw) -> Kara:
    """128 x 16384 decoded tokens, 256-token window (32 protected), chunk budget 64,
    then a keep-20% prune of [2048, 6144)."""
    base = dict(name="kara_prune", B=128, Hq=32, Hkv=8, D=128, page_size=16, ctx=16384,
                dtype=torch.bfloat16, window=256, protected=32, candidates=32, budget=64,
                chunk_coef=0.01, prune_L=2048, prune_R=6144, prune_keep_frac=0.2)
    base.update(kw)
    return Kara(**base)


def kara_schedule(**kw) -> KaraSchedule:
    """128 sequences decoding 320 steps over 2048 + window tokens, 32/8 heads,
    d=128, bf16; Kara window 256 (32 protected), candidates 32, chunk budget
    64, compressions staggered over the 160-step period."""
    base = dict(name="kara_schedule", B=128, Hq=32, Hkv=8, D=128, page_size=16, ctx=2304,
                dtype=torch.bfloat16, window=256, protected=32, candidates=32, budget=64,
                chunk_coef=0.01, steps=320)
    base.update(kw)
    return KaraSchedule(**base)


WORKLOADS = {
    "snapkv_tiny": snapkv_tiny,
    "snapkv_llama8b": snapkv_llama8b,
    "quest_decode": quest_decode,
    "h2o_decode": h2o_decode,
    "kara_prune": kara_prune,
    "kara_schedule": kara_schedule,
}


# ----------------------------------------------------------------------------
# Paged cache construction
# ----------------------------------------------------------------------------


def cdiv(a: int, b: int) -> int:
    return (a + b - 1) // b


@dataclasses.dataclass
class PagedCache:
    """Tensors of one paged KV cache in the library's layout.

    k_pool, v_pool : [num_pages][Hkv][page_size][D]   (dtype)
    block_table    : [B][max_pages_per_seq] int32      physical page id, -1 = none
    slot_map       : [B][Hkv][max_pages_per_seq*page_size] int32  logical position
                     held by each resident slot, -1 beyond ctx_len
    ctx_len        : [B] int32   resident entries per KV head (equal across heads)
    logical_len    : [B] int32   logical prefix length
    free_list      : [num_pages] int32 stack of free page ids, valid below free_top
    free_top       : [1] int32
    page_refcount  : [num_pages] int32 (1 for pages in use, 0 for free pages)
    status         : [1] int32   device error word (0 = ok)
    """
    k_pool: torch.Tensor
    v_pool: torch.Tensor
    block_table: torch.Tensor
    slot_map: torch.Tensor
    ctx_len: torch.Tensor
    logical_len: torch.Tensor
    free_list: torch.Tensor
    free_top: torch.Tensor
    page_refcount: torch.Tensor
    status: torch.Tensor
    page_size: int

    @property
    def B(self):
        return self.block_table.shape[0]

    @property
    def Hkv(self):
        return self.k_pool.shape[1]

    @property
    def D(self):
        return self.k_pool.shape[3]

    @property
    def num_pages(self):
        return self.k_pool.shape[0]

    @property
    def max_pages_per_seq(self):
        return self.block_table.shape[1]

    def clone(self) -> "PagedCache":
        return PagedCache(**{f.name: (getattr(self, f.name).clone()
                                      if isinstance(getattr(self, f.name), torch.Tensor)
                                      else getattr(self, f.name))
                             for f in dataclasses.fields(self)})

    def to(self, device) -> "PagedCache":
        return PagedCache(**{f.name: (getattr(self, f.name).to(device)
                                      if isinstance(getattr(self, f.name), torch.Tensor)
                                      else getattr(self, f.name))
                             for f in dataclasses.fields(self)})


def build_paged_cache(shape: Shape, *, num_pages: int, max_ctx: int, device,
                      tag: str = "cache", ctx: Optional[int] = None) -> PagedCache:
    """Fill ``ctx`` resident tokens per sequence with N(0,1) K/V in scattered pages.

    Slot i of sequence b holds logical position i (a cache right after prefill
    or after plain decoding).  Pages are taken from a seeded permutation of the
    pool; the rest of the pool is the free list.
    """
    ctx = shape.ctx if ctx is None else ctx
    P, B, Hkv, D = shape.page_size, shape.B, shape.Hkv, shape.D
    maxp = cdiv(max_ctx, P)
    used = cdiv(ctx, P)
    if used * B > num_pages:
        raise ValueError("pool too small")
    perm = torch.randperm(num_pages, generator=generator("cpu", shape.name, tag, "pages"))
    perm = perm.to(torch.int32)
    bt = torch.full((B, maxp), -1, dtype=torch.int32)
    bt[:, :used] = perm[: used * B].view(B, used)
    free = torch.zeros(num_pages, dtype=torch.int32)
    nfree = num_pages - used * B
    free[:nfree] = perm[used * B:]
    refc = torch.zeros(num_pages, dtype=torch.int32)
    refc[perm[: used * B].long()] = 1
    slot_map = torch.full((B, Hkv, maxp * P), -1, dtype=torch.int32)
    slot_map[:, :, :ctx] = torch.arange(ctx, dtype=torch.int32)
    k_pool = torch.zeros((num_pages, Hkv, P, D), dtype=shape.dtype, device=device)
    v_pool = torch.zeros((num_pages, Hkv, P, D), dtype=shape.dtype, device=device)
    bt_dev = bt.to(device)
    # Per-sequence draws so that any one sequence can be re-drawn on its own.
    for b in range(B):
        kb = normal((used, Hkv, P, D), shape.dtype, device, shape.name, tag, "k", b)
        vb = normal((used, Hkv, P, D), shape.dtype, device, shape.name, tag, "v", b)
        tail = used * P - ctx          # slots past ctx in the last page stay zero
        if tail:
            kb[-1, :, P - tail:, :] = 0
            vb[-1, :, P - tail:, :] = 0
        pages = bt_dev[b, :used].long()
        k_pool[pages] = kb
        v_pool[pages] = vb
    return PagedCache(
        k_pool=k_pool, v_pool=v_pool, block_table=bt_dev,
        slot_map=slot_map.to(device),
        ctx_len=torch.full((B,), ctx, dtype=torch.int32, device=device),
        logical_len=torch.full((B,), ctx, dtype=torch.int32, device=device),
        free_list=free.to(device),
        free_top=torch.tensor([nfree], dtype=torch.int32, device=device),
        page_refcount=refc.to(device),
        status=torch.zeros(1, dtype=torch.int32, device=device),
        page_size=P)


def slot_to_page(cache: PagedCache, b: int, slot: int):
    return int(cache.block_table[b, slot // cache.page_size]), slot % cache.page_size


# ----------------------------------------------------------------------------
# Heavy keys
# ----------------------------------------------------------------------------


def plant_heavy_keys(shape: SnapKV, cache: PagedCache, tag: str = "cache") -> dict:
    """Make some scored-prefix keys stand out, as the workload text describes.

    Returns {(b, h): positions} of the modified keys (for reporting only).
    """
    P = shape.page_size
    out = {}
    n_scored = shape.scored
    for b in range(shape.B):
        for h in range(shape.Hkv):
            if shape.heavy_mode == "scale4":
                pos = choose(n_scored, shape.heavy_count, shape.name, tag, "heavy", b, h)
            else:
                cnt = int(math.floor(0.01 * n_scored))
                pos = choose(n_scored, cnt, shape.name, tag, "heavy", b, h)
            pages = cache.block_table[b, (pos // P).to(cache.block_table.device)].long()
            rows = (pos % P).to(pages.device)
            k = cache.k_pool[pages, h, rows, :].float()
            if shape.heavy_mode == "scale4":
                k = k * 4.0
            else:
                u = normal((shape.D,), torch.float64, "cpu", shape.name, tag, "dir", b, h)
                u = (u / torch.linalg.vector_norm(u)).to(torch.float32).to(k.device)
                k = k + 3.0 * u
            cache.k_pool[pages, h, rows, :] = k.to(shape.dtype)
            out[(b, h)] = pos
    return out


# ----------------------------------------------------------------------------
# Per-workload inputs
# ----------------------------------------------------------------------------


def snapkv_inputs(shape: SnapKV, device, *, spare_pages: Optional[int] = None):
    """Cache + window queries + one decode query per sequence."""
    P = shape.page_size
    per_seq = cdiv(shape.ctx, P)
    fresh = cdiv(shape.budget, P)
    spare = fresh * shape.B if spare_pages is None else spare_pages
    cache = build_paged_cache(shape, num_pages=per_seq * shape.B + spare,
                              max_ctx=shape.ctx, device=device)
    plant_heavy_keys(shape, cache)
    q_win = normal((shape.B, shape.window, shape.Hq, shape.D), shape.dtype, device,
                   shape.name, "q_win")
    q_pos = (torch.arange(shape.window, dtype=torch.int32) + shape.scored).repeat(shape.B, 1)
    q_dec = normal((shape.B, shape.Hq, shape.D), shape.dtype, device, shape.name, "q_dec")
    return dict(cache=cache, q_win=q_win, q_pos=q_pos.to(device), q_dec=q_dec)


def quest_inputs(shape: Quest, device):
    P = shape.page_size
    per_seq = cdiv(shape.ctx, P)
    cache = build_paged_cache(shape, num_pages=per_seq * shape.B, max_ctx=shape.ctx,
                              device=device)
    q_steps = normal((shape.steps, shape.B, shape.Hq, shape.D), shape.dtype, device,
                     shape.name, "q_steps")
    return dict(cache=cache, q_steps=q_steps)


def h2o_inputs(shape: H2O, device, *, steps: Optional[int] = None):
    P = shape.page_size
    steps = shape.steps if steps is None else steps
    per_seq = cdiv(shape.ctx, P)
    fresh = cdiv(shape.budget + 1, P) + 1
    cache = build_paged_cache(shape, num_pages=(per_seq + fresh) * shape.B,
                              max_ctx=shape.ctx + steps, device=device)
    q_prompt = normal((shape.B, shape.ctx, shape.Hq, shape.D), shape.dtype, device,
                      shape.name, "q_prompt")
    q_pos = torch.arange(shape.ctx, dtype=torch.int32).repeat(shape.B, 1).to(device)
    q_steps = normal((steps, shape.B, shape.Hq, shape.D), shape.dtype, device,
                     shape.name, "q_steps")
    k_steps = normal((steps, shape.B, shape.Hkv, shape.D), shape.dtype, device,
                     shape.name, "k_steps")
    v_steps = normal((steps, shape.B, shape.Hkv, shape.D), shape.dtype, device,
                     shape.name, "v_steps")
    return dict(cache=cache, q_prompt=q_prompt, q_pos=q_pos, q_steps=q_steps,
                k_steps=k_steps, v_steps=v_steps)


def h2o_chunked_inputs(shape: H2O, chunk: int, device):
    """Chunk-wise prefill of the H2O prompt: an empty cache, and the prompt's
    queries, keys and values laid out chunk-major ([n_chunks][B][chunk]...),
    so that each chunk is one contiguous block.  The pool holds the largest
    resident set (budget + chunk) plus the fresh pages of one compaction."""
    if shape.ctx % chunk:
        raise ValueError("the prompt must be a whole number of chunks")
    P = shape.page_size
    n = shape.ctx // chunk
    per_seq = cdiv(shape.budget + chunk, P) + cdiv(shape.budget, P) + 1
    cache = build_paged_cache(shape, num_pages=per_seq * shape.B,
                              max_ctx=shape.budget + chunk, device=device, ctx=0,
                              tag="chunked")
    q = normal((n, shape.B, chunk, shape.Hq, shape.D), shape.dtype, device, shape.name,
               "chunked", "q")
    k = normal((n, shape.B, chunk, shape.Hkv, shape.D), shape.dtype, device, shape.name,
               "chunked", "k")
    v = normal((n, shape.B, chunk, shape.Hkv, shape.D), shape.dtype, device, shape.name,
               "chunked", "v")
    pos = torch.arange(shape.ctx, dtype=torch.int32).view(n, 1, chunk).repeat(1, shape.B, 1)
    return dict(cache=cache, q_chunks=q, k_chunks=k, v_chunks=v, q_pos=pos.to(device))


def kara_schedule_inputs(shape: KaraSchedule, device, *, steps: Optional[int] = None):
    """ctx resident tokens per sequence; sequence b's uncompressed window is its
    last shape.fill(b) slots.  q_ring holds the queries of the last `window`
    logical positions (slot position % window); per-step q, k, v."""
    P = shape.page_size
    steps = shape.steps if steps is None else steps
    max_ctx = shape.ctx + steps + P
    per_seq = cdiv(max_ctx, P) + cdiv(shape.window, P) + 1
    cache = build_paged_cache(shape, num_pages=per_seq * shape.B, max_ctx=max_ctx,
                              device=device)
    q_ring = normal((shape.B, shape.window, shape.Hq, shape.D), shape.dtype, device,
                    shape.name, "q_ring")
    q_steps = normal((steps, shape.B, shape.Hq, shape.D), shape.dtype, device, shape.name,
                     "q_steps")
    k_steps = normal((steps, shape.B, shape.Hkv, shape.D), shape.dtype, device, shape.name,
                     "k_steps")
    v_steps = normal((steps, shape.B, shape.Hkv, shape.D), shape.dtype, device, shape.name,
                     "v_steps")
    return dict(cache=cache, q_ring=q_ring, q_steps=q_steps, k_steps=k_steps, v_steps=v_steps)


def kara_inputs(shape: Kara, device):
    P = shape.page_size
    per_seq = cdiv(shape.ctx, P)
    win_fresh = cdiv(shape.budget + shape.protected, P)
    span_pages = cdiv(shape.ctx, P) - shape.prune_L // P
    spare = (win_fresh + span_pages) * shape.B
    cache = build_paged_cache(shape, num_pages=per_seq * shape.B + spare,
                              max_ctx=shape.ctx, device=device)
    q_win = normal((shape.B, shape.window, shape.Hq, shape.D), shape.dtype, device,
                   shape.name, "q_win")
    q_pos = (torch.arange(shape.window, dtype=torch.int32)
             + (shape.ctx - shape.window)).repeat(shape.B, 1).to(device)
    span = shape.prune_R - shape.prune_L
    mask = torch.zeros((shape.B, span), dtype=torch.uint8)
    for b in range(shape.B):
        mask[b, choose(span, shape.prune_keep, shape.name, "prune_mask", b)] = 1
    q_dec = normal((shape.B, shape.Hq, shape.D), shape.dtype, device, shape.name, "q_dec")
    return dict(cache=cache, q_win=q_win, q_pos=q_pos, prune_mask=mask.to(device),
                q_dec=q_dec)
