"""CPU oracle for attention-scored sparse KV selection, eviction and decode.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import, call or
execute this package: only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` use it.  It shares
no code with the CUDA library (``attention_scored_sparse_gb300``); both read
the seeded tensors that ``se_workloads`` builds.

Every function is a plain, slow, obviously correct restatement of what the
pages define, in fp64 (inputs are bf16/fp32 values widened exactly), written
in the pages' order and notation:

* ``scoring``   window scoring (softmax of Q_win K^T / sqrt(d), summed over the
                GQA group and the window queries) and avg-pooling
                -- SparseEngine "How it works" (finish_step hooks for SnapKV /
                H2O); KARA Method section 1 (sliding-window bidirectional
                attention scoring).
* ``selection`` per-KV-head top-k with forced ranges, Kara Token2Chunk, H2O
                evict-one -- SparseEngine "How it works"; KARA Method
                sections 1-2.
* ``cache``     paged cache model: physical compaction into fresh pages,
                move-last eviction, append, prefix-span pruning
                R' = (R \\ T) U I -- SparseEngine "How it works" (physical
                eviction updates slot mapping and context length and returns
                slots to the allocator) and "How it differs" (prefix pruning,
                idle blocks only).
* ``quest``     per-page key min/max metadata and the page upper bound
                sum_i max(q_i kmax_i, q_i kmin_i) -- SparseEngine "What it is" /
                "How it works" (Quest query-dependent page selection).
* ``attention`` o = Attention(q, BuildView(C, I)) over dense, page-list or
                token-list views -- SparseEngine "How it works" (AttentionView).
* ``pipelines`` the five workloads end to end.

Readings where the pages are silent are marked "reading (n)" at the place they
are taken; the same numbering is used in the design notes.  Functions whose
result rests only on such a reading say "parity unpinned" for that part.
"""
from . import cache, scoring, selection, quest, attention, pipelines  # noqa: F401
