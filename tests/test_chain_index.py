"""Chain index (SparseEngine "How it differs", Chain Cache): the native index
against the reference model, on hand-worked cases and random operation
sequences (CPU only: the index is host code)."""
import random

import pytest

import __graft_entry__

__graft_entry__._builder().build()
import attention_scored_sparse_gb300 as se  # noqa: E402
from oracle.chain_index import ChainIndex as Model  # noqa: E402


def test_model_hand_worked_resume_and_lru_reclaim():
    m = Model(2)
    assert m.acquire([1, 2]) == (1, 0, 0, -1)          # new chain, lowest free row
    assert m.acquire([5]) == (2, 1, 0, -1)
    assert m.finish(1, [1, 2, 3])
    assert m.finish(2, [5, 6])
    # longest idle prefix of the request wins; it is resumed on its own row
    assert m.acquire([1, 2, 3, 4]) == (1, 0, 3, -1)
    # a prefix that does not match is never resumed; all rows taken -> the
    # least recently used idle chain (2) is reclaimed
    assert m.acquire([7, 7]) == (3, 1, 0, 1)
    assert m.acquire([9]) == (0, -1, 0, -1)            # both rows busy: refused
    assert m.finish(3, [7, 7, 8])
    assert m.drop(3) == 1 and m.drop(3) == -1


def test_model_ties_prefer_most_recent():
    m = Model(3)
    assert m.acquire([1]) == (1, 0, 0, -1)
    assert m.acquire([1]) == (2, 1, 0, -1)             # chain 1 is busy: a new chain
    m.finish(1, [1])
    m.finish(2, [1])
    # two idle chains with prefix [1]: the one finished last (2) is resumed
    assert m.acquire([1, 5]) == (2, 1, 1, -1)
    # [1] is no prefix of []: a new chain on the free row
    assert m.acquire([]) == (3, 2, 0, -1)
    # no match, no free row: the only idle chain (1) gives up its row
    assert m.acquire([3]) == (4, 0, 0, 0)


def _same(native, model, op):
    assert native == model, op


@pytest.mark.parametrize("seed", range(6))
def test_native_index_matches_model_on_random_sessions(seed):
    rng = random.Random(seed)
    n_rows = rng.choice([1, 2, 4, 7])
    nat, mod = se.ChainIndex(n_rows), Model(n_rows)
    busy = {}
    vocab = [1, 2, 3]
    for step in range(400):
        r = rng.random()
        if r < 0.45 or not busy:
            base = list(rng.choice(list(busy.values()) or [[]])) if busy and rng.random() < 0.3 else []
            toks = base + [rng.choice(vocab) for _ in range(rng.randint(0, 4))]
            want = mod.acquire(toks)
            if want[0] == 0:
                with pytest.raises(se.SEError):
                    nat.acquire(toks)
                continue
            got = nat.acquire(toks)
            _same(got, want, ("acquire", step, toks))
            busy[got[0]] = toks
        elif r < 0.9:
            cid = rng.choice(list(busy))
            toks = busy.pop(cid) + [rng.choice(vocab) for _ in range(rng.randint(0, 3))]
            assert mod.finish(cid, toks)
            nat.finish(cid, toks)
        else:
            idle = [c for c in mod.chains if not mod.chains[c]["busy"]]
            if not idle:
                continue
            cid = rng.choice(idle)
            _same(nat.drop(cid), mod.drop(cid), ("drop", step))
        assert len(nat) == len(mod.chains)


def test_native_index_rejects_bad_calls():
    ix = se.ChainIndex(1)
    cid, row, reuse, rec = ix.acquire([4, 5])
    with pytest.raises(se.SEError):
        ix.drop(cid)                                   # busy chains are not dropped
    with pytest.raises(se.SEError):
        ix.finish(cid + 7, [1])                        # unknown id
    ix.finish(cid, [4, 5])
    with pytest.raises(se.SEError):
        ix.finish(cid, [4, 5])                         # already idle
    assert ix.drop(cid) == row
    assert len(ix) == 0
    assert se._lib.se_chain_index_create(0) is None
