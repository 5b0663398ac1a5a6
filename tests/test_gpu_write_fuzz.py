"""Seeded random quantize-on-write configurations against the oracle, bit for bit (GPU).

Each case draws a format (int8 side, int8 inline, E4M3), token type (bf16, fp16), head dim,
KV-head count, token count, pool size, a slot mapping with skipped (-1) and out-of-range
entries, zero and outlier tokens, and either slot ids or a paged pool (block table, sequence
and position per token). Stored codes and scales must equal the oracle's bytes; out-of-range
entries are flagged and change nothing. ("int8 per-(token,head) KV cache for the
Qwen3.8-Flash-Next QSA path" §The finding worth upstreaming; "Qwen3.8 Flash Next NVFP4 QSA FP8
E4M3 KV Scales" §Calibration.)
"""

import numpy as np
import pytest
import torch

from gen import f32_to_bf16_bits, f32_to_f16_bits
from oracle import quant as oq

pytestmark = pytest.mark.gpu


def _draw(seed):
    rng = np.random.default_rng([7351, seed])
    return dict(fmt=str(rng.choice(["int8_side", "int8_inline", "e4m3"])), act=str(rng.choice(["bf16", "f16"])),
                hd=int(rng.choice([128, 256])), hkv=int(rng.choice([1, 2, 4])), T=int(rng.integers(1, 3000)),
                extra=int(rng.integers(0, 3000)), skip=float(rng.choice([0.0, 0.1])),
                bad=bool(rng.integers(2)), paged=bool(rng.integers(3) == 0), block=int(rng.choice([1, 16, 12])),
                seed=int(rng.integers(1 << 30)))


@pytest.mark.parametrize("case", range(48))
def test_random_write(case):
    import quantized_kv_cache_write_gb300 as q
    c = _draw(case)
    rng = np.random.default_rng(c["seed"])
    T, H, D = c["T"], c["hkv"], c["hd"]
    x = rng.standard_normal((2, T, H, D), dtype=np.float32)
    x[:, rng.random(T) < 0.02] *= 16.0                       # outlier tokens
    x[:, rng.random(T) < 0.01] = 0.0                         # all-zero tokens (scale 0)
    bits = f32_to_bf16_bits(x) if c["act"] == "bf16" else f32_to_f16_bits(x)
    kb, vb = bits[0], bits[1]
    S = T + c["extra"]
    fmt = {"int8_side": q.QKV_INT8_SIDE, "int8_inline": q.QKV_INT8_INLINE, "e4m3": q.QKV_E4M3}[c["fmt"]]
    dt = torch.float16 if c["act"] == "f16" else torch.bfloat16
    tok = lambda b: torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(dt).cuda()
    # where each token goes: distinct slots, some skipped, some out of range (flagged)
    slots = rng.permutation(S)[:T].astype(np.int64)
    slots[rng.random(T) < c["skip"]] = -1
    kw = {}
    if c["paged"]:
        B = c["block"]
        nblk = (S + B - 1) // B
        nseq = 3
        per = (nblk + nseq - 1) // nseq
        table = np.full((nseq, per), -1, dtype=np.int32)
        perm = rng.permutation(nblk)
        for j in range(nblk):
            table[j % nseq, j // nseq] = perm[j]
        seq = rng.integers(0, nseq, T).astype(np.int32)
        pos = rng.integers(0, per * B, T).astype(np.int32)
        pos[rng.random(T) < c["skip"]] = -1
        # the slot each (sequence, position) names: block_table[seq, pos / B] * B + pos % B
        slots = np.full(T, -1, dtype=np.int64)
        for t in range(T):
            if pos[t] >= 0:
                blk = table[seq[t], pos[t] // B]
                s = int(blk) * B + pos[t] % B
                slots[t] = s if (blk >= 0 and s < S) else -2  # -2: flagged, skipped
        # keep one writer per slot (the oracle and the kernel would race on duplicates)
        seen = set()
        for t in range(T):
            if slots[t] >= 0:
                if slots[t] in seen:
                    pos[t], slots[t] = -1, -1
                seen.add(int(slots[t]))
        kw = dict(token_seq=torch.from_numpy(seq).cuda(), token_pos=torch.from_numpy(pos).cuda(),
                  block_table=torch.from_numpy(table).cuda(), block_size=B)
        expect_flag = bool((slots == -2).any())
    else:
        expect_flag = False
        if c["bad"]:
            slots[rng.integers(0, T)] = S + int(rng.integers(0, 5))
            expect_flag = True
        kw = dict(slot_mapping=torch.from_numpy(slots).cuda())
    oracle_slots = np.where(slots >= S, -1, np.where(slots < -1, -1, slots))
    oracle_slots = np.where(oracle_slots < 0, -1, oracle_slots)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    rec = D + 4 if c["fmt"] == "int8_inline" else D
    kc = torch.zeros((S, H, rec), dtype=torch.uint8, device="cuda")
    vc = torch.zeros_like(kc)
    ks = vs = None
    if c["fmt"] == "int8_side":
        ks = torch.zeros((S, H), dtype=torch.float32, device="cuda")
        vs = torch.zeros_like(ks)
    kscale = vscale = 1.0
    if c["fmt"] == "e4m3":
        kscale = float(oq.e4m3_calibrated_scale(kb, dtype=c["act"]))
        vscale = float(oq.e4m3_calibrated_scale(vb, dtype=c["act"]))
        kscale = kscale if kscale > 0 else 1.0
        vscale = vscale if vscale > 0 else 1.0
    q.qkv_write_ex(tok(kb), tok(vb), fmt, kc, vc, k_scale=ks, v_scale=vs, k_scale_layer=kscale,
                   v_scale_layer=vscale, dev_status=status, **kw)
    torch.cuda.synchronize()
    assert (status.item() & q.QKV_DEV_BAD_SLOT != 0) == expect_flag, c
    if c["fmt"] == "e4m3":
        ref = oq.write_e4m3(kb, vb, oracle_slots, S, np.float32(kscale), np.float32(vscale), dtype=c["act"])
        got = [kc, vc]
    else:
        ref = oq.write_int8(kb, vb, oracle_slots, S, "side" if c["fmt"] == "int8_side" else "inline", dtype=c["act"])
        got = [kc, vc] + ([ks, vs] if c["fmt"] == "int8_side" else [])
    for g, r in zip(got, ref):
        assert g.cpu().numpy().view(np.uint8).tobytes() == np.ascontiguousarray(r).view(np.uint8).tobytes(), c
