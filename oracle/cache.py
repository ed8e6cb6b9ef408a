"""Paged KV cache model for the oracle (test infrastructure only).

SparseEngine, "How it works": the CacheManager owns KV representation,
physical layout, position mapping and the allocate / write / update / free
operations; *physical eviction* rewrites the retained slot mapping and the
context length and hands discarded slots back to the allocator, while
*logical selection* only changes which resident entries attention reads.
SparseEngine, "How it differs": prefix pruning of an application span
[L, R) keeps the logical prefix P and changes only the resident position set,
R' = (R \\ T) U I, freeing the slots that leave R'; the mask is applied to idle
blocks only (no active reference, no transfer in flight).

The pages fix no layout, allocator order or placement; the readings taken here:

reading (xii)  fresh pages are popped from the top of the free-list stack in
               order of ascending sequence, then ascending block index; old
               pages are pushed afterwards in the same order.  Survivors keep
               their order.  All pops of one call happen before its pushes.
reading (ix')  move-last eviction: the entry in the last resident slot moves
               into the victim slot and the context shrinks by one; a page that
               becomes empty is pushed to the free list.
reading (xvii) a page whose reference count is above one is "busy": pruning
               keeps every entry in it, and compaction drops this sequence's
               reference (count - 1) instead of pushing it to the free list.

K/V are held as raw bit patterns (uint16 for bf16, uint32 for fp32) so that
every data movement here is bit-exact; ``values`` widens them to fp64.

All functions update the Cache in place and return a status.  ``seqs``
(optional) limits the K/V data movement to those sequences -- page, slot-map
and free-list bookkeeping is always done for every sequence -- so that a
full-size cache can be checked on a sample of sequences.
"""
from __future__ import annotations

import dataclasses
from typing import List, Optional, Sequence

import numpy as np

SE_OK = 0
SE_ERR_OUT_OF_PAGES = 3
SE_ERR_UNEVEN = 4
SE_ERR_BOUNDS = 7


def cdiv(a: int, b: int) -> int:
    return -(-a // b)


def values(bits: np.ndarray) -> np.ndarray:
    """Widen bf16 (uint16) or fp32 (uint32) bit patterns exactly to fp64."""
    if bits.dtype == np.uint16:
        return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    if bits.dtype == np.uint32:
        return bits.view(np.float32).astype(np.float64)
    raise TypeError(bits.dtype)


@dataclasses.dataclass
class Cache:
    k: np.ndarray            # [num_pages][Hkv][P][D] raw bits
    v: np.ndarray
    block_table: np.ndarray  # [B][maxp] int64, -1 = none
    slot_map: np.ndarray     # [B][Hkv][maxp*P] int64 logical position, -1 = none
    ctx_len: np.ndarray      # [B]
    logical_len: np.ndarray  # [B]
    free_list: np.ndarray    # [num_pages]
    free_top: int
    page_refcount: np.ndarray  # [num_pages]
    page_size: int

    @property
    def B(self):
        return self.block_table.shape[0]

    @property
    def Hkv(self):
        return self.k.shape[1]

    @property
    def D(self):
        return self.k.shape[3]

    def copy(self) -> "Cache":
        return Cache(**{f.name: (getattr(self, f.name).copy()
                                 if isinstance(getattr(self, f.name), np.ndarray)
                                 else getattr(self, f.name))
                        for f in dataclasses.fields(self)})

    # -- addressing --------------------------------------------------------
    def where(self, b: int, slots):
        """(page, row) arrays of resident slots of sequence b."""
        slots = np.asarray(slots, dtype=np.int64)
        P = self.page_size
        pages = self.block_table[b, slots // P]
        assert (pages >= 0).all(), "slot outside the block table"
        return pages, slots % P

    def keys(self, b: int, h: int, slots) -> np.ndarray:
        p, r = self.where(b, slots)
        return values(self.k[p, h, r, :])

    def vals(self, b: int, h: int, slots) -> np.ndarray:
        p, r = self.where(b, slots)
        return values(self.v[p, h, r, :])


def _bits(t):
    import torch
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16).copy()
    if t.dtype == torch.float32:
        return t.view(torch.int32).numpy().view(np.uint32).copy()
    raise TypeError(t.dtype)


def _ints(t):
    return t.detach().cpu().numpy().astype(np.int64)


def from_tensors(pc, seqs: Optional[Sequence[int]] = None, blocks=None) -> Cache:
    """Snapshot a ``se_workloads.PagedCache`` (torch tensors) as an oracle Cache.

    With ``seqs`` only the pages of those sequences are copied (plus, for
    every sequence, the pages of the block range ``blocks`` = (lo, hi)); the
    other pages stay zero (lazily allocated), which is enough for checks
    restricted to those sequences / blocks.
    """
    bt = _ints(pc.block_table)
    if seqs is None:
        k, v = _bits(pc.k_pool), _bits(pc.v_pool)
    else:
        shape = tuple(pc.k_pool.shape)
        dt = np.uint16 if str(pc.k_pool.dtype) == "torch.bfloat16" else np.uint32
        k = np.zeros(shape, dtype=dt)
        v = np.zeros(shape, dtype=dt)
        import torch
        want = [bt[b][bt[b] >= 0] for b in seqs]
        if blocks is not None:
            want += [bt[b, blocks[0]:blocks[1]] for b in range(bt.shape[0])]
        pages = np.unique(np.concatenate(want))
        pages = pages[pages >= 0]
        for i in range(0, len(pages), 4096):
            part = pages[i:i + 4096]
            idx = torch.as_tensor(part, device=pc.k_pool.device)
            k[part] = _bits(pc.k_pool.index_select(0, idx))
            v[part] = _bits(pc.v_pool.index_select(0, idx))
    return Cache(k=k, v=v, block_table=bt, slot_map=_ints(pc.slot_map),
                 ctx_len=_ints(pc.ctx_len), logical_len=_ints(pc.logical_len),
                 free_list=_ints(pc.free_list), free_top=int(pc.free_top.reshape(-1)[0]),
                 page_refcount=_ints(pc.page_refcount), page_size=pc.page_size)


# ---------------------------------------------------------------------------
# Physical compaction (SparseEngine "How it works": physical eviction)
# ---------------------------------------------------------------------------


def compact(c: Cache, keep: List[List[np.ndarray]], first_slot: Sequence[int],
            aux: Optional[np.ndarray] = None, seqs=None) -> int:
    """Rewrite every sequence from page floor(first_slot/P) on, into fresh pages.

    keep[b][h]: ascending resident slots in [first_slot[b], ctx_len[b]) that
    survive; all heads of a sequence keep the same number.  New resident slots
    of sequence b: [0, first_slot) unchanged (those sharing the first
    rewritten page are copied into the fresh page at the same slot), then
    keep[b][h] in order.  Slots past the new length get position -1 (aux 0).
    A sequence with first_slot = ctx_len and nothing kept is left untouched.
    On SE_ERR_OUT_OF_PAGES / SE_ERR_UNEVEN nothing changes.
    """
    P = c.page_size
    B, H = c.B, c.Hkv
    n_keep = []
    for b in range(B):
        counts = {len(keep[b][h]) for h in range(H)}
        if len(counts) != 1:
            return SE_ERR_UNEVEN
        n_keep.append(counts.pop())

    # Page accounting: every pop (ascending b, then block) before any push.
    # Reading (xxv): a sequence whose rewrite is empty (first_slot = ctx_len,
    # nothing kept) is left as it is -- no page moves.
    untouched = [int(first_slot[b]) == int(c.ctx_len[b]) and n_keep[b] == 0 for b in range(B)]
    first_block = [cdiv(int(c.ctx_len[b]), P) if untouched[b] else first_slot[b] // P
                   for b in range(B)]
    new_ctx = [first_slot[b] + n_keep[b] for b in range(B)]
    n_new = [max(cdiv(new_ctx[b], P) - first_block[b], 0) for b in range(B)]
    old_blocks = [cdiv(int(c.ctx_len[b]), P) for b in range(B)]
    if sum(n_new) > c.free_top:
        return SE_ERR_OUT_OF_PAGES

    top = c.free_top
    fresh = []
    for b in range(B):
        fresh.append([int(c.free_list[top - 1 - i]) for i in range(n_new[b])])
        top -= n_new[b]

    old_bt = c.block_table.copy()
    for b in range(B):
        pb, old_ctx = first_block[b], int(c.ctx_len[b])
        head = np.arange(pb * P, first_slot[b], dtype=np.int64)
        dst = np.arange(pb * P, new_ctx[b], dtype=np.int64)
        dst_page = np.array(fresh[b], dtype=np.int64)[(dst - pb * P) // P] if len(dst) else dst
        for h in range(H):
            kh = np.asarray(keep[b][h], dtype=np.int64)
            assert ((kh >= first_slot[b]) & (kh < old_ctx)).all(), "keep slot out of range"
            assert (np.diff(kh) > 0).all(), "keep slots must ascend"
            src = np.concatenate([head, kh])
            if seqs is None or b in seqs:
                sp = old_bt[b, src // P]
                c.k[dst_page, h, dst % P, :] = c.k[sp, h, src % P, :]
                c.v[dst_page, h, dst % P, :] = c.v[sp, h, src % P, :]
            row = c.slot_map[b, h].copy()
            c.slot_map[b, h, dst] = row[src]
            c.slot_map[b, h, new_ctx[b]:old_ctx] = -1
            if aux is not None:
                arow = aux[b, h].copy()
                aux[b, h, dst] = arow[src]
                aux[b, h, new_ctx[b]:old_ctx] = 0.0
        for i, page in enumerate(fresh[b]):
            c.block_table[b, pb + i] = page
        c.block_table[b, pb + n_new[b]: old_blocks[b]] = -1
        c.ctx_len[b] = new_ctx[b]

    refc = c.page_refcount.copy()
    for b in range(B):
        for page in fresh[b]:
            c.page_refcount[page] = 1
    for b in range(B):
        for blk in range(first_block[b], old_blocks[b]):
            page = int(old_bt[b, blk])
            if refc[page] > 1:                  # busy: drop this sequence's reference
                c.page_refcount[page] = refc[page] - 1
            else:
                c.page_refcount[page] = 0
                c.free_list[top] = page
                top += 1
    c.free_top = top
    return SE_OK


def move_last(c: Cache, victim: np.ndarray, aux: Optional[np.ndarray] = None) -> int:
    """H2O physical eviction of one entry per (sequence, KV head).

    victim[b][h]: slot to evict, or -1 on every head of a sequence that evicts
    nothing.  reading (ix'): the last resident slot's entry (data, position,
    aux score) moves into the victim slot; ctx_len shrinks by one; a page left
    empty is pushed to the free list (ascending b).
    """
    P = c.page_size
    for b in range(c.B):
        vs = victim[b]
        if (vs < 0).all():
            continue
        if (vs < 0).any():
            return SE_ERR_UNEVEN
    for b in range(c.B):
        vs = victim[b]
        if (vs < 0).all():
            continue
        last = int(c.ctx_len[b]) - 1
        (sp,), (sr,) = c.where(b, [last])
        for h in range(c.Hkv):
            v = int(vs[h])
            assert 0 <= v <= last
            if v != last:
                (dp,), (dr,) = c.where(b, [v])
                c.k[dp, h, dr, :] = c.k[sp, h, sr, :]
                c.v[dp, h, dr, :] = c.v[sp, h, sr, :]
                c.slot_map[b, h, v] = c.slot_map[b, h, last]
                if aux is not None:
                    aux[b, h, v] = aux[b, h, last]
            c.slot_map[b, h, last] = -1
            if aux is not None:
                aux[b, h, last] = 0.0
        c.ctx_len[b] = last
        if last % P == 0:
            page = int(c.block_table[b, last // P])
            c.block_table[b, last // P] = -1
            c.page_refcount[page] = 0
            c.free_list[c.free_top] = page
            c.free_top += 1
    return SE_OK


def append(c: Cache, k_bits: np.ndarray, v_bits: np.ndarray,
           aux: Optional[np.ndarray] = None) -> int:
    """CacheManager "write": one new token per sequence at slot ctx_len.

    k_bits, v_bits: [B][Hkv][D] raw bits.  A sequence whose last page is full
    takes a fresh page (popped in ascending b).  The new slot holds logical
    position logical_len; both lengths grow by one; aux (if any) starts at 0.
    """
    P = c.page_size
    need = [b for b in range(c.B) if c.ctx_len[b] % P == 0]
    if len(need) > c.free_top:
        return SE_ERR_OUT_OF_PAGES
    for b in range(c.B):
        s = int(c.ctx_len[b])
        if s % P == 0:
            c.free_top -= 1
            page = int(c.free_list[c.free_top])
            c.block_table[b, s // P] = page
            c.page_refcount[page] = 1
        page = int(c.block_table[b, s // P])
        c.k[page, :, s % P, :] = k_bits[b]
        c.v[page, :, s % P, :] = v_bits[b]
        c.slot_map[b, :, s] = c.logical_len[b]
        if aux is not None:
            aux[b, :, s] = 0.0
        c.ctx_len[b] = s + 1
        c.logical_len[b] += 1
    return SE_OK


def append_tokens(c: Cache, k_bits: np.ndarray, v_bits: np.ndarray,
                  aux: Optional[np.ndarray] = None) -> int:
    """CacheManager "write" of n tokens per sequence (a prefill chunk).

    k_bits, v_bits: [B][n][Hkv][D] raw bits.  Token i of sequence b goes to
    slot ctx_len[b] + i with logical position logical_len[b] + i.  Every block
    that was empty before takes a fresh page; all fresh pages are popped from
    the free-list top in ascending (sequence, block) order, as compaction
    pops them (reading xii).  For one sequence this is the same as n
    single-token appends.  Nothing changes on an error.
    """
    P = c.page_size
    n = int(k_bits.shape[1])
    cap = c.block_table.shape[1] * P
    if any(int(c.ctx_len[b]) + n > cap for b in range(c.B)):
        return SE_ERR_BOUNDS
    need = sum(cdiv(int(c.ctx_len[b]) + n, P) - cdiv(int(c.ctx_len[b]), P) for b in range(c.B))
    if need > c.free_top:
        return SE_ERR_OUT_OF_PAGES
    for b in range(c.B):
        ctx = int(c.ctx_len[b])
        for blk in range(cdiv(ctx, P), cdiv(ctx + n, P)):
            c.free_top -= 1
            page = int(c.free_list[c.free_top])
            c.block_table[b, blk] = page
            c.page_refcount[page] = 1
        for i in range(n):
            s = ctx + i
            page = int(c.block_table[b, s // P])
            c.k[page, :, s % P, :] = k_bits[b, i]
            c.v[page, :, s % P, :] = v_bits[b, i]
            c.slot_map[b, :, s] = c.logical_len[b] + i
            if aux is not None:
                aux[b, :, s] = 0.0
        c.ctx_len[b] = ctx + n
        c.logical_len[b] += n
    return SE_OK


def release(c: Cache, mask: Sequence[int]) -> int:
    """CacheManager "free" of whole sequences (SparseEngine "How it differs":
    idle chains are reclaimed when capacity is needed).

    Every sequence b with mask[b] != 0 gives back all its pages: in
    ascending (sequence, block) order each page is pushed onto the free list,
    except a page whose reference count is above one, which only loses this
    sequence's reference (reading xvii).  Reading (xxiv): counts are judged
    as they were before the call, so a page shared by two sequences released
    in the same call loses both references and is pushed by neither; callers
    release such sequences in separate calls.  The block table and slot map
    of a released sequence become -1 and both lengths 0.
    """
    before = c.page_refcount.copy()
    for b in range(c.B):
        if not mask[b]:
            continue
        for blk in range(c.block_table.shape[1]):
            page = int(c.block_table[b, blk])
            if page < 0:
                continue
            if before[page] > 1:
                c.page_refcount[page] -= 1
            else:
                c.page_refcount[page] = 0
                c.free_list[c.free_top] = page
                c.free_top += 1
            c.block_table[b, blk] = -1
        c.slot_map[b] = -1
        c.ctx_len[b] = 0
        c.logical_len[b] = 0
    return SE_OK


# ---------------------------------------------------------------------------
# Prefix-span pruning (SparseEngine "How it differs")
# ---------------------------------------------------------------------------


def prune_plan(c: Cache, L: Sequence[int], R: Sequence[int], mask: np.ndarray):
    """Keep lists for R' = (R \\ T) U I with T = [L, R) and I = {t in T : mask}.

    The pages' "R" is the resident position set (called Res here, apart from
    the span bound R).  Per head: Res'_h = (Res_h \\ T) U (I n Res_h); an entry
    in a busy page (refcount > 1) is kept whatever the mask says (idle blocks
    only).  The rewrite starts at the first resident slot, over all heads,
    whose position is >= L.  mask[b][t - L[b]] is 1 for t in I.

    Returns (status, keep, first_slot, busy_pages) where busy_pages[b] counts
    the busy pages of the rewritten region.
    """
    P = c.page_size
    keep, first, busy = [], [], []
    for b in range(c.B):
        ctx = int(c.ctx_len[b])
        pos = c.slot_map[b, :, :ctx]                          # [H][ctx]
        at_or_after = np.nonzero((pos >= L[b]).any(axis=0))[0]
        fs = int(at_or_after[0]) if len(at_or_after) else ctx
        first.append(fs)
        slots = np.arange(fs, ctx)
        page_busy = c.page_refcount[c.block_table[b, slots // P]] > 1
        busy.append(int(sum(c.page_refcount[c.block_table[b, blk]] > 1
                            for blk in range(fs // P, cdiv(ctx, P)))))
        kb = []
        for h in range(c.Hkv):
            p = pos[h, fs:ctx]
            in_T = (p >= L[b]) & (p < R[b])
            in_I = np.zeros_like(in_T)
            in_I[in_T] = mask[b, p[in_T] - L[b]] != 0
            leaves = in_T & ~in_I & ~page_busy
            kb.append(slots[~leaves].astype(np.int64))
        if len({len(x) for x in kb}) != 1:
            return SE_ERR_UNEVEN, None, None, None
        keep.append(kb)
    return SE_OK, keep, first, busy


def prune(c: Cache, L, R, mask, aux=None, seqs=None):
    """Prune plan, then compaction from the first rewritten page."""
    st, keep, first, busy = prune_plan(c, L, R, mask)
    if st != SE_OK:
        return st, None
    st = compact(c, keep, first, aux, seqs=seqs)
    return st, busy
