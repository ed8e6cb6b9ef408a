"""Reference model of the chain index (test infrastructure only).

SparseEngine "How it differs" (Chain Cache): a session is tied to its
retained KV, its method state and its logical token prefix; because eviction
never changes the logical prefix, a later request whose tokens start with a
chain's prefix resumes from that chain's retained KV and prefills only the
remaining suffix.  Every session has a chain_id; idle chains are reclaimed
least-recently-used first when capacity is needed.

Readings (the pages fix no more than the above):
  (xxi)  a chain occupies one sequence row of the paged cache; a request
         resumes the idle chain with the LONGEST logical prefix that is a
         prefix of its tokens (ties: the most recently used); a chain whose
         prefix is not a prefix of the request is never resumed.
  (xxii) with no chain to resume, a free row is taken (lowest row first); if
         none is free, the least recently used idle chain is reclaimed and
         its row reused; if every row is busy the request is refused.
  (xxiii) "use" is acquire and finish; chain ids count up from 1.
"""
from __future__ import annotations

from typing import Dict, List, Optional, Sequence, Tuple


class ChainIndex:
    def __init__(self, n_rows: int):
        self.n_rows = n_rows
        self.rows: List[Optional[int]] = [None] * n_rows     # row -> chain id
        self.chains: Dict[int, dict] = {}                     # id -> {row, tokens, busy, used}
        self.next_id = 1
        self.clock = 0

    def _tick(self) -> int:
        self.clock += 1
        return self.clock

    def acquire(self, tokens: Sequence[int]) -> Tuple[int, int, int, int]:
        """Returns (chain_id, row, reuse_len, reclaimed_row); reclaimed_row is
        the row whose old chain was dropped (-1 if none); chain_id 0 means
        refused (every row busy)."""
        tokens = list(tokens)
        best = None
        for cid, ch in self.chains.items():
            if ch["busy"]:
                continue
            n = len(ch["tokens"])
            if n <= len(tokens) and tokens[:n] == ch["tokens"]:
                key = (n, ch["used"])
                if best is None or key > best[0]:
                    best = (key, cid)
        if best is not None:
            cid = best[1]
            ch = self.chains[cid]
            ch["busy"] = True
            ch["used"] = self._tick()
            return cid, ch["row"], len(ch["tokens"]), -1
        reclaimed = -1
        free = [r for r in range(self.n_rows) if self.rows[r] is None]
        if free:
            row = free[0]
        else:
            idle = [(ch["used"], cid) for cid, ch in self.chains.items() if not ch["busy"]]
            if not idle:
                return 0, -1, 0, -1
            _, victim = min(idle)
            row = self.chains[victim]["row"]
            del self.chains[victim]
            reclaimed = row
        cid = self.next_id
        self.next_id += 1
        self.chains[cid] = {"row": row, "tokens": [], "busy": True, "used": self._tick()}
        self.rows[row] = cid
        return cid, row, 0, reclaimed

    def finish(self, cid: int, tokens: Sequence[int]) -> bool:
        """The request on chain cid ended; its logical prefix is now tokens."""
        ch = self.chains.get(cid)
        if ch is None or not ch["busy"]:
            return False
        ch["tokens"] = list(tokens)
        ch["busy"] = False
        ch["used"] = self._tick()
        return True

    def drop(self, cid: int) -> int:
        """Forgets an idle chain; returns its row (-1 if unknown or busy)."""
        ch = self.chains.get(cid)
        if ch is None or ch["busy"]:
            return -1
        del self.chains[cid]
        self.rows[ch["row"]] = None
        return ch["row"]
