"""Paged slot pools: logical token positions -> slot ids through a block table.

TEST INFRASTRUCTURE ONLY (see oracle/__init__.py).

[E4M3-PR] "[Model][SM70][FP8] Add calibrated E4M3 QSA KV cache" §Implementation scope: the
KV reads run over paged ("page4") storage. The pages fix no interface; this follows the usual
vLLM block table: sequence s's logical position p lives in block block_table[s, p // B] at
offset p % B, i.e. slot = block_table[s, p // B] * B + p % B for block size B.

What counts as invalid (flagged, then read as padding) is the library's stated contract:
p < -1, p >= max_blocks * B, an unallocated block (id < 0), a slot >= num_slots, and a row
whose sequence lies outside [0, num_seqs) (the whole row is then empty).
"""

import numpy as np


def paged_slots(block_table, row_seq, topk_pos, block_size, num_slots):
    """Translate positions to slot ids.

    Returns (slots int64 [R, k] with -1 for padding and invalid entries,
             bad bool [R, k] marking the entries that are invalid, not merely padding,
             bad_row bool [R] marking rows whose sequence is out of range).
    """
    block_table = np.asarray(block_table, dtype=np.int64)
    row_seq = np.asarray(row_seq, dtype=np.int64)
    pos = np.asarray(topk_pos, dtype=np.int64)
    num_seqs, max_blocks = block_table.shape
    B = int(block_size)
    R, k = pos.shape
    slots = np.full((R, k), -1, dtype=np.int64)
    bad = np.zeros((R, k), dtype=bool)
    bad_row = (row_seq < 0) | (row_seq >= num_seqs)
    for r in range(R):
        if bad_row[r]:
            continue
        for j in range(k):
            p = int(pos[r, j])
            if p == -1:
                continue
            if p < -1 or p >= max_blocks * B:
                bad[r, j] = True
                continue
            blk = int(block_table[row_seq[r], p // B])
            slot = blk * B + p % B
            if blk < 0 or slot >= num_slots:
                bad[r, j] = True
                continue
            slots[r, j] = slot
    return slots, bad, bad_row
