"""The library's C++ block manager (pkv_bm_*) against the oracle block manager.

Both follow the same reading (lowest free page first, forks share every
page, copy-on-write of a shared last page), so seeded random sequences of
add / fork / append / free must give identical slots, copy pairs, block
tables, reference counts and free counts; failures must leave both
unchanged.  Host only: no GPU.
"""
import numpy as np
import pytest

import paged_kv_cache_225_gb300 as pkv
from oracle.block_manager import BlockManager as OracleBM, BlockManagerError

B = 16
NO_BLOCKS, INVALID = 7, 1


def _same_state(bm, ob, live, max_blocks):
    assert bm.num_free() == ob.num_free()
    for b in range(ob.num_blocks):
        assert bm.ref_count(b) == ob.ref[b]
    if live:
        tab, lens = bm.tables(sorted(live), max_blocks)
        for row, ln, seq in zip(tab, lens, sorted(live)):
            t = ob.table(seq)
            assert list(row[:len(t)]) == t and np.all(row[len(t):] == -1)
            assert ln == ob.length(seq)


@pytest.mark.parametrize("seed", range(6))
def test_random_operations_match_the_oracle(seed):
    rng = np.random.default_rng(100 + seed)
    N, max_blocks = 48, 8
    bm, ob = pkv.BlockManager(N, B, max_blocks), OracleBM(N, B, max_blocks)
    live, next_id = set(), 0
    for _ in range(500):
        op = rng.integers(0, 10)
        ids = sorted(live)
        if op < 2 or not ids:
            n = int(rng.integers(0, 70))
            try:
                want = ob.add(next_id, n)
            except BlockManagerError:
                with pytest.raises(pkv.PkvError):
                    bm.add(next_id, n)
            else:
                assert list(bm.add(next_id, n)) == want
                live.add(next_id)
            next_id += 1
        elif op < 4:
            parent = int(rng.choice(ids))
            ob.fork(parent, next_id)
            bm.fork(parent, next_id)
            live.add(next_id)
            next_id += 1
        elif op < 9:
            batch = [int(x) for x in rng.choice(ids, size=min(len(ids), int(rng.integers(1, 5))),
                                                replace=False)]
            # The oracle appends one at a time; a batch that cannot complete
            # must be refused as a whole by the library.
            snapshot = (list(ob.free), list(ob.ref), {k: list(v) for k, v in ob.tables.items()},
                        dict(ob.lens))
            try:
                want = [ob.append(s) for s in batch]
            except BlockManagerError:
                ob.free, ob.ref, ob.tables, ob.lens = snapshot
                import heapq
                heapq.heapify(ob.free)
                with pytest.raises(pkv.PkvError) as e:
                    bm.append(batch)
                assert e.value.code in (NO_BLOCKS, INVALID)
            else:
                slots, pairs = bm.append(batch)
                assert list(slots) == [w[0] for w in want]
                assert [tuple(p) for p in pairs] == [c for w in want for c in w[1]]
        else:
            s = int(rng.choice(ids))
            ob.free_seq(s)
            bm.free(s)
            live.discard(s)
        _same_state(bm, ob, live, max_blocks)


def test_errors_change_nothing():
    bm = pkv.BlockManager(4, B, 3)
    bm.add(0, 40)                                    # 3 pages
    with pytest.raises(pkv.PkvError) as e:
        bm.add(0, 1)                                 # duplicate id
    assert e.value.code == INVALID
    with pytest.raises(pkv.PkvError) as e:
        bm.add(1, 40)                                # 3 pages, 1 free
    assert e.value.code == NO_BLOCKS
    with pytest.raises(pkv.PkvError) as e:
        bm.add(2, 49)                                # 4 pages > 3 per sequence
    assert e.value.code == INVALID
    with pytest.raises(pkv.PkvError):
        bm.fork(5, 6)                                # unknown parent
    with pytest.raises(pkv.PkvError):
        bm.append([0, 0])                            # listed twice
    with pytest.raises(pkv.PkvError):
        bm.free(9)
    assert bm.num_free() == 1
    tab, lens = bm.tables([0], 3)
    assert list(lens) == [40] and list(tab[0]) == [0, 1, 2]


def test_batched_append_counts_a_shared_page_once():
    # Two forks share a partly filled last page; with one free page the
    # batch still fits: the first copies, the second then writes in place.
    bm = pkv.BlockManager(3, B, 4)
    bm.add(0, 20)                                    # pages 0, 1 (1 holds 4 tokens)
    bm.fork(0, 1)
    slots, pairs = bm.append([0, 1])
    assert [tuple(p) for p in pairs] == [(1, 2)]
    assert list(slots) == [2 * B + 4, 1 * B + 4]
    assert bm.num_free() == 0
