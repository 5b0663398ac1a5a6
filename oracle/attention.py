"""Oracle top-k gather decode attention in fp64 (test infrastructure; see the package docstring).

What is computed                     [INT8-PR §The finding worth upstreaming: the QSA path
                                      gathers each row's scattered top-k slots]
    For query row r, query head g (KV head h = g // (Hq / Hkv)) and the row's index list
    idx[r, :] (slot ids; -1 entries are padding and skipped):
        J      = the valid entries of idx[r, :], in the given order
        K_j    = dequantised K of slot j, head h (fp64); V_j likewise
        s_j    = softmax_scale * sum_d q[r, g, d] * K_j[d]
        o      = sum_j exp(s_j - max s) V_j / sum_j exp(s_j - max s)
        lse    = max s + log sum_j exp(s_j - max s)          (natural log)
    A row with no valid entry gives o = 0 and lse = -inf.

Dequantisation (per element, the plain definition; the hoisted form is a pin):
    int8 side / inline : K_j[d] = c_j[d] * scale_j           [INT8-PR; INT8-KV]
    E4M3               : K_j[d] = dec(c_j[d]) * k_scale_layer  [SCALES §Calibration]
    bf16               : K_j[d] = the stored bf16 value

Split-K and merge                    [HOIST-PR §Changes; E4M3-PR §Implementation scope]
    Split s of P takes index columns [s*c, min(k, (s+1)*c)) with c = ceil(k / P); empty
    splits are allowed. Each split yields a normalised partial (o_s, lse_s) over its own
    columns; the merge is
        lse = log sum_s exp(lse_s),   o = sum_s exp(lse_s - lse) * o_s
    then times the post-merge V scale. For E4M3 the per-layer V scale is applied once,
    after normalised accumulation, or after the merge when the row is split; the partials
    therefore hold sum_j p_j dec(c_j) / l (no V scale), which is what `e4m3_pool_fp64`
    with `apply_v_scale=False` provides.
"""

from __future__ import annotations

import math

import numpy as np

from .quant import act_bits_to_f32, bf16_bits_to_f32, e4m3_decode, f16_bits_to_f32


# --------------------------------------------------------------------------- dequantisation

def int8_side_pool_fp64(codes: np.ndarray, scale: np.ndarray) -> np.ndarray:
    """codes int8 [S, Hkv, D], scale fp32 [S, Hkv] -> fp64 [S, Hkv, D], c * scale per element."""
    return codes.astype(np.float64) * scale.astype(np.float64)[..., None]


def int8_inline_pool_fp64(records: np.ndarray) -> np.ndarray:
    """records uint8 [S, Hkv, D + 4] -> fp64 [S, Hkv, D]; scale = little-endian fp32 at byte D."""
    D = records.shape[-1] - 4
    codes = np.ascontiguousarray(records[..., :D]).view(np.int8)
    scale = np.ascontiguousarray(records[..., D:]).view("<f4")[..., 0]
    return int8_side_pool_fp64(codes, scale)


def e4m3_pool_fp64(codes: np.ndarray, scale, apply_scale: bool = True) -> np.ndarray:
    """codes uint8 [S, Hkv, D] -> fp64 dec(c) * scale (or dec(c) alone)."""
    vals = e4m3_decode(codes)
    return vals * float(np.float32(scale)) if apply_scale else vals


def bf16_pool_fp64(bits: np.ndarray) -> np.ndarray:
    return bf16_bits_to_f32(bits).astype(np.float64)


def f16_pool_fp64(bits: np.ndarray) -> np.ndarray:
    """Unquantised fp16 pool (the FP16-activation contract's baseline cache) -> fp64."""
    return f16_bits_to_f32(bits).astype(np.float64)


# --------------------------------------------------------------------------- attention

def _row_attention(qr: np.ndarray, K: np.ndarray, V: np.ndarray, sel: np.ndarray,
                   softmax_scale: float, group: int):
    """One row: qr [Hq, D] fp64, K/V [S, Hkv, D] fp64, sel = valid slot ids. Returns o, lse."""
    Hq, D = qr.shape
    o = np.zeros((Hq, D), dtype=np.float64)
    lse = np.full(Hq, -np.inf, dtype=np.float64)
    if sel.size == 0:
        return o, lse
    Hkv = K.shape[1]
    for h in range(Hkv):
        Kj = K[sel, h, :]  # [n, D]
        Vj = V[sel, h, :]
        qg = qr[h * group:(h + 1) * group]  # [G, D]
        s = softmax_scale * (qg @ Kj.T)  # [G, n]
        m = np.max(s, axis=1, keepdims=True)
        w = np.exp(s - m)
        l = np.sum(w, axis=1, keepdims=True)
        o[h * group:(h + 1) * group] = (w @ Vj) / l
        lse[h * group:(h + 1) * group] = (m + np.log(l))[:, 0]
    return o, lse


def gather_attention(q_bits: np.ndarray, K: np.ndarray, V: np.ndarray, topk: np.ndarray,
                     softmax_scale: float, rows=None, col_range=None, q_dtype: str = "bf16"):
    """Top-k gather attention over a dequantised pool.

    q_bits: uint16 bf16 (or fp16, q_dtype='f16') [R, Hq, D]; K, V: fp64 [S, Hkv, D];
    topk: int [R, k] (-1 = pad).
    rows: optional iterable of row ids to compute (others left at 0 / -inf).
    col_range: optional (a, b) restricting each row to index columns [a, b).
    Returns o fp64 [R, Hq, D] and lse fp64 [R, Hq].
    """
    R, Hq, D = q_bits.shape
    S, Hkv, _ = K.shape
    group = Hq // Hkv
    q = act_bits_to_f32(q_bits, q_dtype).astype(np.float64)
    o = np.zeros((R, Hq, D), dtype=np.float64)
    lse = np.full((R, Hq), -np.inf, dtype=np.float64)
    row_ids = range(R) if rows is None else rows
    a, b = (0, topk.shape[1]) if col_range is None else col_range
    for r in row_ids:
        cols = np.asarray(topk[r, a:b], dtype=np.int64)
        sel = cols[cols >= 0]
        o[r], lse[r] = _row_attention(q[r], K, V, sel, softmax_scale, group)
    return o, lse


def split_bounds(k: int, num_splits: int):
    """Column ranges of the P splits: contiguous chunks of ceil(k / P), the last one shorter."""
    c = -(-k // num_splits) if k > 0 else 0
    return [(min(k, s * c), min(k, (s + 1) * c)) for s in range(num_splits)]


def gather_attention_splits(q_bits, K, V, topk, softmax_scale, num_splits: int, rows=None, q_dtype: str = "bf16"):
    """Per-split normalised partials: o_part [R, P, Hq, D], lse_part [R, P, Hq]."""
    R, Hq, D = q_bits.shape
    o_part = np.zeros((R, num_splits, Hq, D), dtype=np.float64)
    lse_part = np.full((R, num_splits, Hq), -np.inf, dtype=np.float64)
    for s, (a, b) in enumerate(split_bounds(topk.shape[1], num_splits)):
        o_s, l_s = gather_attention(q_bits, K, V, topk, softmax_scale, rows=rows, col_range=(a, b),
                                    q_dtype=q_dtype)
        o_part[:, s] = o_s
        lse_part[:, s] = l_s
    return o_part, lse_part


def merge_splits(o_part: np.ndarray, lse_part: np.ndarray, v_scale_post: float = 1.0):
    """Log-sum-exp merge of split partials, then the post-merge V scale.

    o_part [R, P, Hq, D], lse_part [R, P, Hq] -> o [R, Hq, D], lse [R, Hq].
    All-empty rows (every lse_s = -inf) give o = 0, lse = -inf.
    """
    R, P, Hq, D = o_part.shape
    o = np.zeros((R, Hq, D), dtype=np.float64)
    lse = np.full((R, Hq), -np.inf, dtype=np.float64)
    for r in range(R):
        for g in range(Hq):
            ls = lse_part[r, :, g].astype(np.float64)
            m = np.max(ls)
            if m == -math.inf:
                continue
            w = np.exp(ls - m)
            tot = np.sum(w)
            lse[r, g] = m + math.log(tot)
            o[r, g] = (w / tot) @ o_part[r, :, g, :].astype(np.float64) * float(np.float32(v_scale_post))
    return o, lse
