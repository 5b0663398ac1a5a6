"""Pins of oracle/paging.py (paged pool: logical positions -> slot ids through a block table).

[E4M3-PR] "[Model][SM70][FP8] Add calibrated E4M3 QSA KV cache" §Implementation scope: KV
reads over paged storage. The mapping slot = table[s, p // B] * B + p % B is the usual vLLM
block table (the pages fix no interface).

Pins: a hand-worked table with every invalid case; agreement with the long-context
generator, which places tokens through its own block permutation (independent code); and
planted mistakes that the hand-worked case must catch.
"""

import numpy as np
import pytest

from gen import long_context_decode
from oracle.paging import paged_slots

# block size 4, two sequences of 3 blocks; block ids in units of 4 slots; pool of 18 slots
TABLE = np.array([[3, 0, -1], [1, 2, 4]], dtype=np.int32)
ROW_SEQ = np.array([0, 1, 5], dtype=np.int32)
POS = np.array([[5, 0, 9, -1, 12, -2],
                [11, 4, 3, 7, 8, 1],
                [0, 1, 2, 3, 4, 5]], dtype=np.int32)
# worked by hand:
#   row 0, seq 0: 5 -> block 1 (id 0) -> 1; 0 -> block 0 (id 3) -> 12; 9 -> block 2 (id -1)
#                 unallocated; -1 padding; 12 >= 3 * 4 out of range; -2 invalid
#   row 1, seq 1: 11 -> block 2 (id 4) -> 19 >= 18 past the pool; 4 -> id 2 -> 8; 3 -> id 1
#                 -> 7; 7 -> id 2 -> 11; 8 -> id 4 -> 16; 1 -> id 1 -> 5
#   row 2: sequence 5 of 2 -> the row is empty (not flagged per entry)
SLOTS = np.array([[1, 12, -1, -1, -1, -1],
                  [-1, 8, 7, 11, 16, 5],
                  [-1, -1, -1, -1, -1, -1]])
BAD = np.array([[0, 0, 1, 0, 1, 1],
                [1, 0, 0, 0, 0, 0],
                [0, 0, 0, 0, 0, 0]], dtype=bool)


def test_hand_worked_table():
    slots, bad, bad_row = paged_slots(TABLE, ROW_SEQ, POS, 4, 18)
    assert np.array_equal(slots, SLOTS)
    assert np.array_equal(bad, BAD)
    assert list(bad_row) == [False, False, True]


def test_agrees_with_the_generators_own_placement():
    wl = long_context_decode(seed=5, num_seqs=3, context=4096, rows_per_seq=2, topk=256, recent=512,
                             recent_picks=192, num_splits=1)
    slots, bad, bad_row = paged_slots(wl.block_table, wl.row_seq, wl.topk_pos, wl.block_size, wl.num_slots)
    assert not bad.any() and not bad_row.any()
    assert np.array_equal(slots, wl.topk.astype(np.int64))


def _swapped_offset(table, row_seq, pos, B, S):
    # planted mistake: offset and block index swapped
    s2 = np.full(pos.shape, -1, dtype=np.int64)
    for r in range(pos.shape[0]):
        for j in range(pos.shape[1]):
            p = int(pos[r, j])
            if 0 <= p < table.shape[1] * B and 0 <= row_seq[r] < table.shape[0]:
                blk = int(table[row_seq[r], p % table.shape[1]])
                if blk >= 0 and blk * B + p // table.shape[1] < S:
                    s2[r, j] = blk * B + p // table.shape[1]
    return s2


def _ignores_sequence(table, row_seq, pos, B, S):
    # planted mistake: every row read through sequence 0's table row
    return paged_slots(table, np.zeros_like(row_seq), pos, B, S)[0]


@pytest.mark.parametrize("mistake", [_swapped_offset, _ignores_sequence])
def test_planted_mistakes_are_caught(mistake):
    assert not np.array_equal(mistake(TABLE, ROW_SEQ, POS, 4, 18), SLOTS)
