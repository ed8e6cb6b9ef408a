"""Workload pipelines: the C-ABI calls in the order the methods use them.

Each class preallocates every buffer it needs (scores, kept indices,
workspaces) at construction, so a step launches kernels only and can be
captured in a CUDA graph.  Call order follows the pages: SparseEngine "How it
works" (SnapKV / H2O selection at the end of prefill via finish_step, Quest
selection per decode step via build_decode_selection, physical eviction,
AttentionView) and KARA Method 3 (periodic compression of the trailing
window); SparseEngine "How it differs" (prefix-span pruning).
"""
from __future__ import annotations

import torch

from . import (SE_COMPACT_FRESH_PAGES, SE_COMPACT_MOVE_LAST, SE_SELECT_EVICT_ONE,
               SE_SELECT_KARA_CHUNK, SE_SELECT_TOPK, SE_VIEW_DENSE, SE_VIEW_PAGES,
               SE_VIEW_TOKENS, kv_desc,
               se_append_kv, se_compact_decode, se_compact_evict, se_prune_span,
               se_quest_build_meta,
               se_quest_decode_step, se_quest_page_select, se_score_window,
               se_sparse_decode_attn, se_topk_select,
               workspace_sizes)


def _i32(vals, device):
    return torch.as_tensor(vals, dtype=torch.int32).to(device)


class _Base:
    def __init__(self, cache, Hq):
        self.cache = cache
        self.Hq = Hq
        self.kv = kv_desc(cache, Hq)
        self.device = cache.k_pool.device
        self.B = cache.block_table.shape[0]
        self.Hkv = cache.k_pool.shape[1]
        self.P = cache.page_size
        self.max_slots = cache.slot_map.shape[-1]

    def _ws(self, nbytes):
        # zeroed: the scoring workspace starts with a control block that each
        # call leaves at zero for the next
        return torch.zeros(max(int(nbytes), 256), dtype=torch.uint8, device=self.device)


class _Snapshot:
    """A cache's tensors with the block table and context lengths replaced by
    other tensors (copies taken before compaction rewrites them)."""

    def __init__(self, cache, block_table, ctx_len):
        for n in ("k_pool", "v_pool", "slot_map", "logical_len", "free_list", "free_top",
                  "status", "page_size"):
            setattr(self, n, getattr(cache, n))
        self.page_refcount = getattr(cache, "page_refcount", None)
        self.block_table = block_table
        self.ctx_len = ctx_len


class SnapKV(_Base):
    """SnapKV after the last prompt chunk: causal window scores, avg-pool +
    top-k per KV head with the window forced, compaction into fresh pages,
    then decode attention over the retained entries."""

    def __init__(self, cache, Hq, *, ctx, window, budget, pool_kernel):
        super().__init__(cache, Hq)
        B, dev = self.B, self.device
        self.ctx, self.window, self.budget, self.pool = ctx, window, budget, pool_kernel
        scored = ctx - window
        self.zero = _i32([0] * B, dev)
        self.ctx_t = _i32([ctx] * B, dev)
        self.scored_t = _i32([scored] * B, dev)
        self.scores = torch.zeros((B, self.Hkv, self.max_slots), dtype=torch.float32, device=dev)
        self.keep = torch.empty((B, self.Hkv, budget), dtype=torch.int32, device=dev)
        self.n_keep = torch.empty(B, dtype=torch.int32, device=dev)
        sz = workspace_sizes(self.kv, w=window, n_max=ctx, max_keep=budget, max_entries=budget)
        self.ws_score = self._ws(sz["score_window"])
        self.ws_compact = self._ws(sz["compact_evict"])
        self.ws_decode = self._ws(sz["sparse_decode_attn"])
        self.ws_compact_decode = self._ws(sz["compact_decode"])
        # block table and context lengths as they were before compaction, so
        # decode attention can read the kept entries while compaction moves them
        self.bt_snap = torch.empty_like(cache.block_table)
        self.ctx_snap = torch.empty_like(cache.ctx_len)
        self.kv_snap = kv_desc(_Snapshot(cache, self.bt_snap, self.ctx_snap), Hq)
        self.side = torch.cuda.Stream(device=dev)

    def score(self, q_win, q_pos, stream=None):
        se_score_window(self.kv, q_win, q_pos, self.zero, self.ctx_t, self.zero, self.scored_t,
                        causal=True, accumulate=False, n_max=self.ctx, scores=self.scores,
                        workspace=self.ws_score, stream=stream)

    def select(self, stream=None):
        se_topk_select(self.kv, self.scores, mode=SE_SELECT_TOPK, cand_lo=self.zero,
                       cand_hi=self.scored_t, force_lo=self.scored_t, force_hi=self.ctx_t,
                       keep_idx=self.keep, n_keep=self.n_keep, pool_kernel=self.pool,
                       k=self.budget - self.window, n_max=self.ctx - self.window, stream=stream)

    def compact(self, stream=None):
        se_compact_evict(self.kv, SE_COMPACT_FRESH_PAGES, self.keep, n_keep=self.n_keep,
                         first_slot=self.zero, max_keep=self.budget, workspace=self.ws_compact,
                         stream=stream)

    def decode(self, q, o, stream=None):
        se_sparse_decode_attn(self.kv, q, view=SE_VIEW_DENSE, o=o, max_entries=self.budget,
                              workspace=self.ws_decode, stream=stream)

    def decode_kept(self, q, o, stream=None):
        """Decode attention over the kept entries where they lie before
        compaction: the token view of keep_idx through the snapshot of the
        block table and context lengths.  The same entries, in the same order,
        as the dense view of the compacted cache."""
        se_sparse_decode_attn(self.kv_snap, q, view=SE_VIEW_TOKENS, sel=self.keep,
                              n_sel=self.budget, o=o, max_entries=self.budget,
                              workspace=self.ws_decode, stream=stream)

    def compact_decode(self, q, o, stream=None):
        """Compaction and decode attention side by side: the block table and
        context lengths are copied, decode attention runs on a second stream
        over the kept entries in their old pages while compaction copies them
        into fresh pages (it writes only pages it pops from the free list and
        returns the old ones after the copy; nothing reuses them within the
        step), and the stream waits for both.  ``stream`` is a
        ``torch.cuda.Stream`` (default: the current stream)."""
        main = torch.cuda.current_stream(self.device) if stream is None else stream
        with torch.cuda.stream(main):
            self.bt_snap.copy_(self.cache.block_table)
            self.ctx_snap.copy_(self.cache.ctx_len)
        self.side.wait_stream(main)
        self.decode_kept(q, o, self.side)
        self.compact(main)
        main.wait_stream(self.side)

    def compact_decode_fused(self, q, o, stream=None):
        """Compaction and decode attention in one pass over the kept entries
        (se_compact_decode): each kept K/V row is read once, copied into its
        fresh page and attended there."""
        se_compact_decode(self.kv, self.keep, n_keep=self.n_keep, first_slot=self.zero,
                          max_keep=self.budget, q=q, o=o, max_entries=self.budget,
                          workspace=self.ws_compact_decode, stream=stream)

    def step(self, q_win, q_pos, q_dec, o, stream=None):
        self.score(q_win, q_pos, stream)
        self.select(stream)
        self.compact_decode_fused(q_dec, o, stream)


class QuestDecode(_Base):
    """Quest: per-page key min/max once, then per decode step the page bound,
    top pages + current page, and attention over those pages."""

    def __init__(self, cache, Hq, *, ctx, top_pages):
        super().__init__(cache, Hq)
        B, dev = self.B, self.device
        self.top = top_pages
        self.nblocks = (ctx + self.P - 1) // self.P
        shape = (cache.k_pool.shape[0], self.Hkv, cache.k_pool.shape[3])
        self.kmin = torch.empty(shape, dtype=cache.k_pool.dtype, device=dev)
        self.kmax = torch.empty(shape, dtype=cache.k_pool.dtype, device=dev)
        self.page_idx = torch.empty((B, self.Hkv, top_pages + 1), dtype=torch.int32, device=dev)
        self.n_sel = torch.empty(B, dtype=torch.int32, device=dev)
        sz = workspace_sizes(self.kv, max_blocks=self.nblocks,
                             max_entries=(top_pages + 1) * self.P)
        self.ws_sel = self._ws(sz["quest_page_select"])
        self.ws_decode = self._ws(sz["sparse_decode_attn"])

    def build_meta(self, stream=None):
        se_quest_build_meta(self.kv, self.kmin, self.kmax, stream=stream)

    def select(self, q, stream=None):
        se_quest_page_select(self.kv, self.kmin, self.kmax, q, top_pages=self.top,
                             max_blocks=self.nblocks, page_idx=self.page_idx, n_sel=self.n_sel,
                             workspace=self.ws_sel, stream=stream)

    def decode(self, q, o, stream=None):
        se_sparse_decode_attn(self.kv, q, view=SE_VIEW_PAGES, o=o, sel=self.page_idx,
                              n_sel=self.top + 1, max_entries=(self.top + 1) * self.P,
                              workspace=self.ws_decode, stream=stream)

    def step(self, q, o, stream=None):
        self.select(q, stream)
        self.decode(q, o, stream)

    def step_fused(self, q, o, stream=None):
        """The same step as one launch (bounds, selection and attention)."""
        se_quest_decode_step(self.kv, self.kmin, self.kmax, q, o, top_pages=self.top,
                             page_idx=self.page_idx, n_sel=self.n_sel, stream=stream)


class H2O(_Base):
    """H2O: causal scores of the whole prompt seed the running scores and pick
    the initial heavy hitters (plus the recent tokens); each decode step
    appends, attends over every resident entry while adding its weights to
    the running scores, and evicts the lowest-scoring non-recent entry."""

    def __init__(self, cache, Hq, *, prompt, heavy, recent):
        super().__init__(cache, Hq)
        B, dev = self.B, self.device
        self.prompt, self.heavy, self.recent = prompt, heavy, recent
        self.budget = heavy + recent
        self.zero = _i32([0] * B, dev)
        self.ctx_t = _i32([prompt] * B, dev)
        self.cand_t = _i32([prompt - recent] * B, dev)
        self.acc = torch.zeros((B, self.Hkv, self.max_slots), dtype=torch.float32, device=dev)
        self.keep = torch.empty((B, self.Hkv, self.budget), dtype=torch.int32, device=dev)
        self.n_keep = torch.empty(B, dtype=torch.int32, device=dev)
        self.victim = torch.empty((B, self.Hkv), dtype=torch.int32, device=dev)
        sz = workspace_sizes(self.kv, w=prompt, n_max=prompt, max_keep=self.budget,
                             max_entries=self.budget + 1)
        self.ws_score = self._ws(sz["score_window"])
        self.ws_compact = self._ws(sz["compact_evict"])
        self.ws_decode = self._ws(sz["sparse_decode_attn"])
        self.ws_append = self._ws(sz["append_kv"])

    def prefill(self, q_prompt, q_pos, stream=None):
        self.prefill_score(q_prompt, q_pos, stream)
        self.prefill_select(stream)
        self.prefill_compact(stream)

    def prefill_score(self, q_prompt, q_pos, stream=None):
        """Causal scores of the whole prompt into the running scores."""
        se_score_window(self.kv, q_prompt, q_pos, self.zero, self.ctx_t, self.zero, self.ctx_t,
                        causal=True, accumulate=False, n_max=self.prompt, scores=self.acc,
                        workspace=self.ws_score, stream=stream)

    def prefill_select(self, stream=None):
        """Top ``heavy`` of the non-recent prompt plus the ``recent`` tokens."""
        se_topk_select(self.kv, self.acc, mode=SE_SELECT_TOPK, cand_lo=self.zero,
                       cand_hi=self.cand_t, force_lo=self.cand_t, force_hi=self.ctx_t,
                       keep_idx=self.keep, n_keep=self.n_keep, pool_kernel=1, k=self.heavy,
                       n_max=self.prompt - self.recent, stream=stream)

    def prefill_compact(self, stream=None):
        """Compaction of the kept entries from slot 0, scores moving along."""
        se_compact_evict(self.kv, SE_COMPACT_FRESH_PAGES, self.keep, n_keep=self.n_keep,
                         first_slot=self.zero, max_keep=self.budget, aux=self.acc,
                         workspace=self.ws_compact, stream=stream)

    def step(self, q, k_new, v_new, o, stream=None):
        se_append_kv(self.kv, k_new, v_new, aux=self.acc, workspace=self.ws_append, stream=stream)
        se_sparse_decode_attn(self.kv, q, view=SE_VIEW_DENSE, o=o, max_entries=self.budget + 1,
                              acc_scores=self.acc, workspace=self.ws_decode, stream=stream)
        se_topk_select(self.kv, self.acc, mode=SE_SELECT_EVICT_ONE, keep_idx=self.victim,
                       budget=self.budget, recent=self.recent, stream=stream)
        se_compact_evict(self.kv, SE_COMPACT_MOVE_LAST, self.victim, aux=self.acc,
                         workspace=self.ws_compact, stream=stream)


class H2OChunkedPrefill(_Base):
    """H2O chunk-wise prefill eviction: each prompt chunk is written to the
    cache, its queries score every resident entry causally into the running
    scores (new entries start at 0), and once more than heavy + recent
    entries are resident the top ``heavy`` of the older ones plus the last
    ``recent`` are compacted from slot 0, the scores moving with them."""

    def __init__(self, cache, Hq, *, chunk, heavy, recent):
        super().__init__(cache, Hq)
        B, dev = self.B, self.device
        self.chunk, self.heavy, self.recent = chunk, heavy, recent
        self.budget = heavy + recent
        self.zero = _i32([0] * B, dev)
        self.acc = torch.zeros((B, self.Hkv, self.max_slots), dtype=torch.float32, device=dev)
        self.keep = torch.empty((B, self.Hkv, self.budget), dtype=torch.int32, device=dev)
        self.n_keep = torch.empty(B, dtype=torch.int32, device=dev)
        self.n_max = self.budget + chunk
        sz = workspace_sizes(self.kv, w=chunk, n_max=self.n_max, max_keep=self.budget)
        self.ws_score = self._ws(sz["score_window"])
        self.ws_compact = self._ws(sz["compact_evict"])
        self.ws_append = self._ws(sz["append_kv"])
        self._lens = {}

    def _len(self, n):
        if n not in self._lens:
            self._lens[n] = _i32([n] * self.B, self.device)
        return self._lens[n]

    def chunk_step(self, resident, q_chunk, q_pos, k_chunk, v_chunk, stream=None):
        """One chunk on top of ``resident`` entries per sequence; returns the
        resident count afterwards (known on the host, no sync)."""
        ctx = resident + self.chunk
        ctx_t = self._len(ctx)
        se_append_kv(self.kv, k_chunk, v_chunk, aux=self.acc, workspace=self.ws_append,
                     stream=stream)
        se_score_window(self.kv, q_chunk, q_pos, self.zero, ctx_t, self.zero, ctx_t, causal=True,
                        accumulate=True, n_max=ctx, scores=self.acc, workspace=self.ws_score,
                        stream=stream)
        if ctx <= self.budget:
            return ctx
        cand = self._len(ctx - self.recent)
        se_topk_select(self.kv, self.acc, mode=SE_SELECT_TOPK, cand_lo=self.zero, cand_hi=cand,
                       force_lo=cand, force_hi=ctx_t, keep_idx=self.keep, n_keep=self.n_keep,
                       pool_kernel=1, k=self.heavy, n_max=ctx - self.recent, stream=stream)
        se_compact_evict(self.kv, SE_COMPACT_FRESH_PAGES, self.keep, n_keep=self.n_keep,
                         first_slot=self.zero, max_keep=self.budget, aux=self.acc,
                         workspace=self.ws_compact, stream=stream)
        return self.budget

    def run(self, q_chunks, q_pos, k_chunks, v_chunks, stream=None):
        resident = 0
        for i in range(q_chunks.shape[0]):
            resident = self.chunk_step(resident, q_chunks[i], q_pos[i], k_chunks[i], v_chunks[i],
                                       stream=stream)
        return resident


class KaraSchedule(_Base):
    """Kara periodic compression inside a decode loop, staggered over the batch.

    Each step appends every sequence's token, attends over all resident
    entries, and compresses the trailing window of the sequences whose window
    just filled (bidirectional scores of the window's queries, Token2Chunk,
    compaction from the window start); the other sequences get empty ranges
    and are left untouched by every call.  The window's queries live in a
    ring indexed by logical position modulo the window.  Lengths follow from
    the schedule and are tracked on the host; the per-step ranges reach the
    device through pinned buffers with asynchronous copies, so no step waits
    for the GPU."""

    def __init__(self, cache, Hq, *, ctx, fills, window, protected, candidates, budget,
                 chunk_coef, max_ctx, n_staging=8):
        super().__init__(cache, Hq)
        B, dev = self.B, self.device
        self.window, self.protected = window, protected
        self.candidates, self.budget, self.coef = candidates, budget, chunk_coef
        self.ctx = [ctx] * B                         # resident entries (host mirror)
        self.logical = [ctx] * B                     # logical length (host mirror)
        self.win_start = [ctx - f for f in fills]    # first slot of the window
        self.scores = torch.zeros((B, self.Hkv, self.max_slots), dtype=torch.float32, device=dev)
        self.keep = torch.empty((B, self.Hkv, budget + protected), dtype=torch.int32, device=dev)
        self.n_keep = torch.empty(B, dtype=torch.int32, device=dev)
        # device copies of the step's lengths: [logical, win_lo, ctx, prot_lo]
        self.lens = torch.empty((4, B), dtype=torch.int32, device=dev)
        self.staging = [torch.empty((4, B), dtype=torch.int32).pin_memory()
                        for _ in range(n_staging)]
        self.staged = [None] * n_staging             # event after each buffer's copy
        self.n_steps = 0
        self.rows = torch.arange(B, device=dev)
        self.offs = torch.arange(window, dtype=torch.int32, device=dev) - window
        self.max_ctx = max_ctx
        sz = workspace_sizes(self.kv, w=window, n_max=window, max_keep=budget + protected,
                             max_entries=max_ctx)
        self.ws_score = self._ws(sz["score_window"])
        self.ws_compact = self._ws(sz["compact_evict"])
        self.ws_decode = self._ws(sz["sparse_decode_attn"])
        self.ws_append = self._ws(sz["append_kv"])
        self.compressions = 0

    def _upload(self, rows, stream):
        i = self.n_steps % len(self.staging)
        if self.staged[i] is not None:
            self.staged[i].synchronize()             # the copy that used it has run
        buf = self.staging[i]
        buf.copy_(torch.tensor(rows, dtype=torch.int32))
        self.lens.copy_(buf, non_blocking=True)
        ev = torch.cuda.Event()
        ev.record(stream if stream is not None else torch.cuda.current_stream())
        self.staged[i] = ev

    def step(self, q, k_new, v_new, o, q_ring, stream=None):
        B, W = self.B, self.window
        due = [b for b in range(B) if self.ctx[b] + 1 - self.win_start[b] >= W]
        win_lo = [self.ctx[b] + 1 - W if b in due else self.ctx[b] + 1 for b in range(B)]
        ctx1 = [c + 1 for c in self.ctx]
        prot_lo = [ctx1[b] - self.protected if b in due else ctx1[b] for b in range(B)]
        self._upload([self.logical, win_lo, ctx1, prot_lo], stream)
        self.n_steps += 1
        # the new token's query goes to ring slot (its position % window)
        q_ring[self.rows, (self.lens[0] % W).long()] = q
        se_append_kv(self.kv, k_new, v_new, workspace=self.ws_append, stream=stream)
        se_sparse_decode_attn(self.kv, q, view=SE_VIEW_DENSE, o=o, max_entries=self.max_ctx,
                              workspace=self.ws_decode, stream=stream)
        for b in range(B):
            self.ctx[b] += 1
            self.logical[b] += 1
        if not due:
            return due
        # positions of the window's queries: the last W before the new length
        q_pos = (self.lens[0] + 1)[:, None] + self.offs[None, :]
        lo, hi, plo = self.lens[1], self.lens[2], self.lens[3]
        se_score_window(self.kv, q_ring, q_pos, lo, hi, lo, plo, causal=False,
                        accumulate=False, n_max=W, scores=self.scores, workspace=self.ws_score,
                        stream=stream)
        se_topk_select(self.kv, self.scores, mode=SE_SELECT_KARA_CHUNK, cand_lo=lo, cand_hi=plo,
                       force_lo=plo, force_hi=hi, keep_idx=self.keep, n_keep=self.n_keep,
                       k=self.candidates, chunk_budget=self.budget, chunk_coef=self.coef,
                       n_max=W - self.protected, stream=stream)
        se_compact_evict(self.kv, SE_COMPACT_FRESH_PAGES, self.keep, n_keep=self.n_keep,
                         first_slot=lo, max_keep=self.budget + self.protected,
                         workspace=self.ws_compact, stream=stream)
        for b in due:
            self.ctx[b] = win_lo[b] + self.budget + self.protected
        self.compressions += len(due)
        return due


class Kara(_Base):
    """Kara periodic compression of the trailing window (bidirectional scores
    of the compressible keys, Token2Chunk, compaction from the window start),
    prefix-span pruning, and decode attention over the result."""

    def __init__(self, cache, Hq, *, ctx, window, protected, candidates, budget, chunk_coef):
        super().__init__(cache, Hq)
        B, dev = self.B, self.device
        self.ctx, self.window, self.protected = ctx, window, protected
        self.candidates, self.budget, self.coef = candidates, budget, chunk_coef
        self.win_lo = _i32([ctx - window] * B, dev)
        self.prot_lo = _i32([ctx - protected] * B, dev)
        self.ctx_t = _i32([ctx] * B, dev)
        self.scores = torch.zeros((B, self.Hkv, self.max_slots), dtype=torch.float32, device=dev)
        self.keep = torch.empty((B, self.Hkv, budget + protected), dtype=torch.int32, device=dev)
        self.n_keep = torch.empty(B, dtype=torch.int32, device=dev)
        self.n_busy = torch.empty(B, dtype=torch.int32, device=dev)
        sz = workspace_sizes(self.kv, w=window, n_max=window, max_keep=budget + protected,
                             max_entries=ctx)
        self.ws_score = self._ws(sz["score_window"])
        self.ws_compact = self._ws(sz["compact_evict"])
        self.ws_prune = self._ws(sz["prune_span"])
        self.ws_decode = self._ws(sz["sparse_decode_attn"])

    def score(self, q_win, q_pos, stream=None):
        se_score_window(self.kv, q_win, q_pos, self.win_lo, self.ctx_t, self.win_lo,
                        self.prot_lo, causal=False, accumulate=False, n_max=self.window,
                        scores=self.scores, workspace=self.ws_score, stream=stream)

    def select(self, stream=None):
        se_topk_select(self.kv, self.scores, mode=SE_SELECT_KARA_CHUNK, cand_lo=self.win_lo,
                       cand_hi=self.prot_lo, force_lo=self.prot_lo, force_hi=self.ctx_t,
                       keep_idx=self.keep, n_keep=self.n_keep, k=self.candidates,
                       chunk_budget=self.budget, chunk_coef=self.coef,
                       n_max=self.window - self.protected, stream=stream)

    def compact(self, stream=None):
        se_compact_evict(self.kv, SE_COMPACT_FRESH_PAGES, self.keep, n_keep=self.n_keep,
                         first_slot=self.win_lo, max_keep=self.budget + self.protected,
                         workspace=self.ws_compact, stream=stream)

    def compress(self, q_win, q_pos, stream=None):
        self.score(q_win, q_pos, stream)
        self.select(stream)
        self.compact(stream)

    def prune(self, L, R, mask, stream=None):
        se_prune_span(self.kv, L, R, mask, n_busy=self.n_busy, workspace=self.ws_prune,
                      stream=stream)

    def decode(self, q, o, max_entries=None, stream=None):
        se_sparse_decode_attn(self.kv, q, view=SE_VIEW_DENSE, o=o,
                              max_entries=max_entries or self.ctx, workspace=self.ws_decode,
                              stream=stream)
