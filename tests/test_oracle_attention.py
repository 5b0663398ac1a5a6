"""Pins for the oracle's fp64 top-k gather attention, split-K and merge (CPU only).

Every check compares against something the oracle does not compute itself: torch's
scaled_dot_product_attention in float64 on the special cases where the gather reduces to
dense (or masked dense) attention, closed forms (a single key), brute force over every
subset of a tiny pool, and invariances the pages rely on (index order, split count,
hoisted scales: "[Perf][SM70][FP8] Hoist QSA E4M3 KV scales" §Changes; inline vs side
layout: "int8 per-(token,head) KV cache for the Qwen3.8-Flash-Next QSA path" §The finding
worth upstreaming).
"""

import itertools
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from gen import f32_to_bf16_bits, small_random, tiny
from oracle import attention as att
from oracle import quant


def _sdpa(q64, K, V, sel_mask, scale):
    """Library dense attention, fp64. q64 [Hq, D]; K, V [S, Hkv, D]; sel_mask bool [S]."""
    Hq = q64.shape[0]
    Hkv = K.shape[1]
    G = Hq // Hkv
    k = torch.from_numpy(np.repeat(K.transpose(1, 0, 2), G, axis=0))  # [Hq, S, D]
    v = torch.from_numpy(np.repeat(V.transpose(1, 0, 2), G, axis=0))
    q = torch.from_numpy(q64)[:, None, :]  # [Hq, 1, D]
    mask = torch.from_numpy(sel_mask)[None, None, :].expand(Hq, 1, -1)
    o = F.scaled_dot_product_attention(q, k, v, attn_mask=mask, scale=scale)
    s = (q @ k.transpose(1, 2))[:, 0, :] * scale
    s = s.masked_fill(~torch.from_numpy(sel_mask)[None, :], -math.inf)
    return o[:, 0, :].numpy(), torch.logsumexp(s, dim=1).numpy()


def _pool_side(wl):
    kc, vc, ks, vs = quant.write_int8(wl.k_tokens, wl.v_tokens, wl.slot_mapping, wl.num_slots, "side")
    return att.int8_side_pool_fp64(kc, ks), att.int8_side_pool_fp64(vc, vs)


def test_topk_all_slots_equals_dense_attention():
    wl = tiny(0)
    K, V = _pool_side(wl)
    S = wl.num_slots
    rng = np.random.default_rng(1)
    R = 4
    topk = np.stack([rng.permutation(S) for _ in range(R)]).astype(np.int32)
    q = wl.q[:R]
    o, lse = att.gather_attention(q, K, V, topk, wl.softmax_scale)
    q64 = quant.bf16_bits_to_f32(q).astype(np.float64)
    for r in range(R):
        o_ref, lse_ref = _sdpa(q64[r], K, V, np.ones(S, dtype=bool), wl.softmax_scale)
        assert np.max(np.abs(o[r] - o_ref)) < 1e-12
        assert np.max(np.abs(lse[r] - lse_ref)) < 1e-12


def test_brute_force_every_subset_of_a_tiny_pool():
    wl = small_random(21, num_slots=8, rows=1, topk=8, num_q_heads=4, num_kv_heads=2)
    K, V = _pool_side(wl)
    q64 = quant.bf16_bits_to_f32(wl.q[0]).astype(np.float64)
    for n in range(1, 9):
        for subset in itertools.combinations(range(8), n):
            idx = np.full((1, 8), -1, dtype=np.int32)
            idx[0, :n] = subset[::-1]
            o, lse = att.gather_attention(wl.q[:1], K, V, idx, 0.0625)
            mask = np.zeros(8, dtype=bool)
            mask[list(subset)] = True
            o_ref, lse_ref = _sdpa(q64, K, V, mask, 0.0625)
            assert np.max(np.abs(o[0] - o_ref)) < 1e-12
            assert np.max(np.abs(lse[0] - lse_ref)) < 1e-12


def test_single_key_returns_that_value_row():
    wl = small_random(22, num_slots=16, rows=3, topk=1, num_q_heads=8)
    K, V = _pool_side(wl)
    o, lse = att.gather_attention(wl.q, K, V, wl.topk, wl.softmax_scale)
    q64 = quant.bf16_bits_to_f32(wl.q).astype(np.float64)
    for r in range(3):
        j = wl.topk[r, 0]
        assert np.array_equal(o[r], np.broadcast_to(V[j, 0], o[r].shape))
        assert np.allclose(lse[r], wl.softmax_scale * (q64[r] @ K[j, 0]), rtol=0, atol=1e-12)


def test_empty_row_gives_zero_and_minus_inf():
    wl = small_random(23, num_slots=16, rows=2, topk=4)
    K, V = _pool_side(wl)
    idx = wl.topk.copy()
    idx[1] = -1
    o, lse = att.gather_attention(wl.q, K, V, idx, wl.softmax_scale)
    assert np.all(o[1] == 0) and np.all(lse[1] == -np.inf)
    assert np.all(np.isfinite(lse[0]))


def test_index_order_invariance():
    wl = small_random(24, num_slots=512, rows=4, topk=200, outlier_frac=0.05)
    K, V = _pool_side(wl)
    o1, l1 = att.gather_attention(wl.q, K, V, wl.topk, wl.softmax_scale)
    rng = np.random.default_rng(0)
    perm = np.stack([rng.permutation(wl.topk.shape[1]) for _ in range(4)])
    o2, l2 = att.gather_attention(wl.q, K, V, np.take_along_axis(wl.topk, perm, 1), wl.softmax_scale)
    assert np.max(np.abs(o1 - o2)) < 1e-13 and np.max(np.abs(l1 - l2)) < 1e-12


@pytest.mark.parametrize("P", [2, 8, 13, 200])
def test_split_merge_equals_unsplit(P):
    wl = small_random(25, num_slots=512, rows=3, topk=200, pad_frac=0.2)
    K, V = _pool_side(wl)
    o1, l1 = att.gather_attention(wl.q, K, V, wl.topk, wl.softmax_scale)
    op, lp = att.gather_attention_splits(wl.q, K, V, wl.topk, wl.softmax_scale, P)
    o2, l2 = att.merge_splits(op, lp)
    assert np.max(np.abs(o1 - o2)) < 1e-12 and np.max(np.abs(l1 - l2)) < 1e-12


def test_split_bounds_match_the_partition():
    b = att.split_bounds(2051, 8)
    assert [e - s for s, e in b] == [257] * 7 + [252]
    assert att.split_bounds(5, 8)[-3:] == [(5, 5)] * 3  # empty trailing splits
    assert att.split_bounds(0, 4) == [(0, 0)] * 4


def test_merge_identity_and_all_empty():
    rng = np.random.default_rng(2)
    op = rng.standard_normal((2, 1, 4, 256))
    lp = rng.standard_normal((2, 1, 4))
    o, l = att.merge_splits(op, lp)
    assert np.array_equal(o, op[:, 0]) and np.allclose(l, lp[:, 0], atol=1e-15)
    o, l = att.merge_splits(np.zeros((1, 3, 2, 256)), np.full((1, 3, 2), -np.inf))
    assert np.all(o == 0) and np.all(l == -np.inf)


def test_e4m3_scale_hoisting_equals_per_element_dequant():
    wl = small_random(26, num_slots=256, rows=4, topk=100, outlier_frac=0.05)
    ks = quant.e4m3_calibrated_scale(wl.k_tokens)
    vs = quant.e4m3_calibrated_scale(wl.v_tokens)
    kc, vc = quant.write_e4m3(wl.k_tokens, wl.v_tokens, wl.slot_mapping, wl.num_slots, ks, vs)
    K = att.e4m3_pool_fp64(kc, ks)
    V = att.e4m3_pool_fp64(vc, vs)
    o_plain, l_plain = att.gather_attention(wl.q, K, V, wl.topk, wl.softmax_scale)
    # hoisted: K scale folded into the softmax factor, V scale applied once after accumulation
    Kd = att.e4m3_pool_fp64(kc, ks, apply_scale=False)
    Vd = att.e4m3_pool_fp64(vc, vs, apply_scale=False)
    o_h, l_h = att.gather_attention(wl.q, Kd, Vd, wl.topk, wl.softmax_scale * float(ks))
    assert np.max(np.abs(o_plain - float(vs) * o_h)) < 1e-12
    assert np.max(np.abs(l_plain - l_h)) < 1e-12
    # split-K: V scale once after the merge
    op, lp = att.gather_attention_splits(wl.q, Kd, Vd, wl.topk, wl.softmax_scale * float(ks), 8)
    o_m, l_m = att.merge_splits(op, lp, v_scale_post=float(vs))
    assert np.max(np.abs(o_plain - o_m)) < 1e-12 and np.max(np.abs(l_plain - l_m)) < 1e-12


def test_int8_per_token_scale_hoisting():
    """(q . c_j) * s_j equals q . (c_j * s_j); sum_j p_j s_j c_j equals sum_j p_j (s_j c_j)."""
    wl = small_random(27, num_slots=128, rows=2, topk=64)
    kc, vc, ks, vs = quant.write_int8(wl.k_tokens, wl.v_tokens, wl.slot_mapping, 128, "side")
    q = quant.bf16_bits_to_f32(wl.q).astype(np.float64)
    sel = wl.topk[0]
    s_plain = q[0] @ att.int8_side_pool_fp64(kc, ks)[sel, 0].T
    s_hoist = (q[0] @ kc[sel, 0].astype(np.float64).T) * ks[sel, 0].astype(np.float64)[None]
    assert np.max(np.abs(s_plain - s_hoist)) < 1e-12


def test_inline_and_side_layouts_dequantise_identically():
    wl = small_random(28, num_slots=300, rows=1, topk=4, num_tokens=250)
    kc, vc, ks, vs = quant.write_int8(wl.k_tokens, wl.v_tokens, wl.slot_mapping, 300, "side")
    kr, vr = quant.write_int8(wl.k_tokens, wl.v_tokens, wl.slot_mapping, 300, "inline")
    assert np.array_equal(att.int8_side_pool_fp64(kc, ks), att.int8_inline_pool_fp64(kr))
    assert np.array_equal(att.int8_side_pool_fp64(vc, vs), att.int8_inline_pool_fp64(vr))


@pytest.mark.parametrize("bug", ["no_scale", "wrong_head_group", "v_for_k"])
def test_planted_attention_mistakes_are_caught(bug):
    """A plausible mistake in a copy of the row kernel must fail the dense-attention pin."""
    wl = small_random(29, num_slots=64, rows=1, topk=64, num_q_heads=4, num_kv_heads=2)
    K, V = _pool_side(wl)
    q64 = quant.bf16_bits_to_f32(wl.q[0]).astype(np.float64)
    sel = np.arange(64)
    o = np.zeros((4, 256))
    for g in range(4):
        h = (g % 2) if bug == "wrong_head_group" else g // 2
        Kj = (V if bug == "v_for_k" else K)[sel, h]
        s = (1.0 if bug == "no_scale" else wl.softmax_scale) * (Kj @ q64[g])
        w = np.exp(s - s.max())
        o[g] = w @ V[sel, h] / w.sum()
    o_ref, _ = _sdpa(q64, K, V, np.ones(64, dtype=bool), wl.softmax_scale)
    assert np.max(np.abs(o - o_ref)) > 1e-6
