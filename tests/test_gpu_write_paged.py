"""Writes through qkv_write_ex: slot ids and paged addressing (GPU).

"[Model][SM70][FP8] Add calibrated E4M3 QSA KV cache" §Implementation scope: the KV cache is
paged storage. A paged write finds token t's slot through the block table,
block_table[seq, pos / B] * B + pos % B, the addressing the paged gather reads. The stored
bytes must equal the oracle's write to the slots that addressing names. Invalid entries are
flagged and skipped, and the slots they would have hit stay untouched.
"""

import numpy as np
import pytest
import torch

from gen import small_random
from oracle import quant as oq

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def q():
    import quantized_kv_cache_write_gb300 as q
    return q


def _paged_case(seed, block_size, num_tokens, num_seqs=6, max_blocks=9):
    """A block table over a pool of physical blocks, tokens at distinct (sequence, position)
    pairs, and a few deliberately invalid entries. Returns the table, the tokens' sequences
    and positions, the expected slot of each token (-1: skipped) and whether it is flagged."""
    rng = np.random.default_rng(seed)
    phys = num_seqs * max_blocks - 5  # fewer physical blocks than table entries: some unallocated
    table = np.full((num_seqs, max_blocks), -1, dtype=np.int32)
    entries = rng.permutation(num_seqs * max_blocks)[:phys]
    table.flat[entries] = rng.permutation(phys).astype(np.int32)
    num_slots = phys * block_size
    big = int(np.nonzero(table.ravel() >= 0)[0][0])
    table.flat[big] = phys + 3  # an allocated block id past the pool: its slots are out of range
    cand = [(s, p) for s in range(num_seqs) for p in range(max_blocks * block_size)]
    pick = rng.choice(len(cand), num_tokens, replace=False)
    seq = np.array([cand[i][0] for i in pick], dtype=np.int32)
    pos = np.array([cand[i][1] for i in pick], dtype=np.int32)
    # invalid and skipped entries
    seq[0], pos[0] = 0, -1                                  # skipped, not flagged
    pos[1] = max_blocks * block_size                        # past the table
    pos[2] = -5                                             # below -1
    seq[3] = num_seqs                                       # no such sequence
    seq[4] = -1
    expect = np.full(num_tokens, -1, dtype=np.int64)
    flagged = np.zeros(num_tokens, dtype=bool)
    for t in range(num_tokens):
        s, p = int(seq[t]), int(pos[t])
        if p == -1:
            continue
        if p < -1 or p >= max_blocks * block_size or s < 0 or s >= num_seqs:
            flagged[t] = True
            continue
        blk = int(table[s, p // block_size])
        slot = blk * block_size + p % block_size
        if blk < 0 or slot >= num_slots:
            flagged[t] = True
            continue
        expect[t] = slot
    return table, seq, pos, expect, flagged, num_slots


def _bits_dev(bits, act):
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda()
    return t.view(torch.float16 if act == "f16" else torch.bfloat16)


@pytest.mark.parametrize("fmt", ["int8_side", "int8_inline", "e4m3"])
@pytest.mark.parametrize("block_size,act,large", [(16, "bf16", False), (7, "bf16", False), (16, "f16", False),
                                                  (7, "f16", False), (16, "bf16", True)])
def test_paged_write_bit_exact_and_invalid_entries_flagged(q, fmt, block_size, act, large):
    """large: 17000 tokens, past the size where each warp writes a token's K and V rows."""
    if large:
        table, seq, pos, expect, flagged, S = _paged_case(13, block_size, 17000, num_seqs=40, max_blocks=40)
    else:
        table, seq, pos, expect, flagged, S = _paged_case(11 + block_size, block_size, 300)
    assert flagged.any() and (expect >= 0).sum() > 0.8 * len(seq)
    wl = small_random(77, num_slots=S, rows=1, topk=1, num_tokens=len(seq), outlier_frac=0.02, act_dtype=act)
    k, v = _bits_dev(wl.k_tokens, act), _bits_dev(wl.v_tokens, act)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    D = 256
    kw = dict(token_seq=torch.from_numpy(seq).cuda(), token_pos=torch.from_numpy(pos).cuda(),
              block_table=torch.from_numpy(table).cuda(), block_size=block_size, dev_status=status)
    if fmt == "e4m3":
        ks, vs = np.float32(0.0131), np.float32(0.0089)
        kc = torch.full((S, 1, D), 0x5A, dtype=torch.uint8, device="cuda")
        vc = kc.clone()
        q.qkv_write_ex(k, v, q.QKV_E4M3, kc, vc, k_scale_layer=float(ks), v_scale_layer=float(vs), **kw)
        ref = oq.write_e4m3(wl.k_tokens, wl.v_tokens, expect, S, ks, vs, dtype=act)
        got = [kc, vc]
    elif fmt == "int8_side":
        kc = torch.full((S, 1, D), 0x5A, dtype=torch.int8, device="cuda")
        vc = kc.clone()
        ksc = torch.full((S, 1), -1.0, dtype=torch.float32, device="cuda")
        vsc = ksc.clone()
        q.qkv_write_ex(k, v, q.QKV_INT8_SIDE, kc, vc, k_scale=ksc, v_scale=vsc, **kw)
        ref = oq.write_int8(wl.k_tokens, wl.v_tokens, expect, S, "side", dtype=act)
        got = [kc, vc, ksc, vsc]
    else:
        kc = torch.full((S, 1, D + 4), 0x5A, dtype=torch.uint8, device="cuda")
        vc = kc.clone()
        q.qkv_write_ex(k, v, q.QKV_INT8_INLINE, kc, vc, **kw)
        ref = oq.write_int8(wl.k_tokens, wl.v_tokens, expect, S, "inline", dtype=act)
        got = [kc, vc]
    torch.cuda.synchronize()
    assert status.item() == q.QKV_DEV_BAD_SLOT
    written = expect[expect >= 0]
    untouched = np.setdiff1d(np.arange(S), written)
    for g, r in zip(got, ref):
        g = g.cpu().numpy()
        assert g[written].tobytes() == np.ascontiguousarray(r)[written].view(g.dtype).tobytes()
        fill = -1.0 if g.dtype == np.float32 else 0x5A
        assert np.all(g[untouched].view(np.uint8 if g.dtype != np.float32 else np.float32) == fill)


def test_slot_id_write_through_the_descriptor_matches_the_plain_call(q):
    wl = small_random(5, num_slots=40000, rows=1, topk=1, num_tokens=20000, num_kv_heads=1)
    k, v = _bits_dev(wl.k_tokens, "bf16"), _bits_dev(wl.v_tokens, "bf16")
    sm = torch.from_numpy(wl.slot_mapping).cuda()
    a = [torch.zeros((40000, 1, 256), dtype=torch.int8, device="cuda") for _ in range(2)]
    b = [torch.zeros((40000, 1, 256), dtype=torch.int8, device="cuda") for _ in range(2)]
    sa = [torch.zeros((40000, 1), dtype=torch.float32, device="cuda") for _ in range(2)]
    sb = [torch.zeros((40000, 1), dtype=torch.float32, device="cuda") for _ in range(2)]
    q.qkv_write_int8(k, v, sm, a[0], a[1], sa[0], sa[1])
    q.qkv_write_ex(k, v, q.QKV_INT8_SIDE, b[0], b[1], slot_mapping=sm, k_scale=sb[0], v_scale=sb[1])
    torch.cuda.synchronize()
    for x, y in zip(a + sa, b + sb):
        assert torch.equal(x, y)
