"""Test-side helpers: move generator outputs to the GPU, run the library through its C ABI,
run the oracle on the same inputs, and compare with the stated tolerance.

The library side and the oracle side never exchange values: each quantises, calibrates
and attends on its own; only the generator's inputs are shared.
"""

from __future__ import annotations

import numpy as np
import torch

from oracle import attention as oatt
from oracle import quant as oq

ATOL = 5e-5  # attention outputs: |gpu - ref| <= ATOL + RTOL * |ref| against the fp64 oracle
RTOL = 1e-3


def bf16_dev(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def act_dev(bits: np.ndarray, act_dtype: str = "bf16") -> torch.Tensor:
    """16-bit activation bits on the device as bf16 or fp16."""
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.view(torch.float16 if act_dtype == "f16" else torch.bfloat16).cuda()


def assert_close(got: np.ndarray, ref: np.ndarray, what: str, atol=ATOL, rtol=RTOL):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    both_inf = np.isinf(ref) & (got == ref)
    with np.errstate(invalid="ignore"):
        err = np.where(both_inf, 0.0, np.abs(got - ref))
    bad = ~(err <= atol + rtol * np.abs(np.where(both_inf, 0.0, ref)))
    if np.any(bad):
        i = np.unravel_index(np.argmax(np.where(bad, err, -1)), err.shape)
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} outside {atol}+{rtol}|ref|; "
                             f"worst at {i}: got {got[i]!r} ref {ref[i]!r}; max abs err {np.nanmax(err):.3e}")
    return float(np.max(err)) if err.size else 0.0


class GpuPool:
    """A slot pool written on the GPU by the library's own write kernels."""

    def __init__(self, wl, fmt: str, dev_status: torch.Tensor | None = None):
        import quantized_kv_cache_write_gb300 as q
        self.fmt = fmt
        self.code = q.FORMATS[fmt]
        self.act = wl.act_dtype
        S, H, D = wl.num_slots, wl.num_kv_heads, wl.head_dim
        self.k_tok = act_dev(wl.k_tokens, wl.act_dtype)
        self.v_tok = act_dev(wl.v_tokens, wl.act_dtype)
        self.slots = torch.from_numpy(wl.slot_mapping).cuda()
        self.k_scale_tok = self.v_scale_tok = None
        self.k_scale_layer = self.v_scale_layer = 1.0
        if fmt in ("bf16", "f16"):
            self.k_cache = torch.zeros((S, H, D), dtype=self.k_tok.dtype, device="cuda")
            self.v_cache = torch.zeros_like(self.k_cache)
            take = self.slots >= 0
            self.k_cache[self.slots[take]] = self.k_tok[take]
            self.v_cache[self.slots[take]] = self.v_tok[take]
        elif fmt == "int8_side":
            self.k_cache = torch.zeros((S, H, D), dtype=torch.int8, device="cuda")
            self.v_cache = torch.zeros_like(self.k_cache)
            self.k_scale_tok = torch.zeros((S, H), dtype=torch.float32, device="cuda")
            self.v_scale_tok = torch.zeros_like(self.k_scale_tok)
            q.qkv_write_int8(self.k_tok, self.v_tok, self.slots, self.k_cache, self.v_cache,
                             self.k_scale_tok, self.v_scale_tok, layout=q.QKV_INT8_SIDE, dev_status=dev_status)
        elif fmt == "int8_inline":
            self.k_cache = torch.zeros((S, H, D + 4), dtype=torch.uint8, device="cuda")
            self.v_cache = torch.zeros_like(self.k_cache)
            q.qkv_write_int8(self.k_tok, self.v_tok, self.slots, self.k_cache, self.v_cache,
                             layout=q.QKV_INT8_INLINE, dev_status=dev_status)
        elif fmt == "e4m3":
            if wl.act_dtype == "f16":  # the calibration statistics give amax / 448 for half tensors
                ks, vs = (np.float32(_calibrated_scale_f16(t)) for t in (self.k_tok, self.v_tok))
            else:
                amax = torch.zeros(1, dtype=torch.int32, device="cuda")
                sc = torch.zeros(2, dtype=torch.float32, device="cuda")
                q.qkv_e4m3_calibrate(self.k_tok, amax, sc[0:1])
                q.qkv_e4m3_calibrate(self.v_tok, amax, sc[1:2])
                ks, vs = sc.cpu().numpy()
            self.k_scale_layer, self.v_scale_layer = np.float32(ks), np.float32(vs)
            self.k_cache = torch.zeros((S, H, D), dtype=torch.uint8, device="cuda")
            self.v_cache = torch.zeros_like(self.k_cache)
            q.qkv_write_e4m3(self.k_tok, self.v_tok, self.slots, self.k_cache, self.v_cache,
                             float(ks), float(vs), dev_status=dev_status)
        else:
            raise ValueError(fmt)

    def attend(self, wl, q_dev=None, idx_dev=None, num_splits: int = 1, with_lse: bool = True,
               dev_status=None):
        """Run qsa_gather_attn (and the merge when split). Returns out, lse (and partials)."""
        import quantized_kv_cache_write_gb300 as q
        qd = act_dev(wl.q, wl.act_dtype) if q_dev is None else q_dev
        idx = torch.from_numpy(np.ascontiguousarray(wl.topk, dtype=np.int32)).cuda() if idx_dev is None else idx_dev
        R, Hq, D = qd.shape
        kw = dict(num_kv_heads=wl.num_kv_heads, num_slots=wl.num_slots, k_scale_tok=self.k_scale_tok,
                  v_scale_tok=self.v_scale_tok, k_scale_layer=float(self.k_scale_layer),
                  v_scale_layer=float(self.v_scale_layer), dev_status=dev_status)
        if num_splits == 1:
            out = torch.full((R, Hq, D), float("nan"), dtype=torch.float32, device="cuda")
            lse = torch.full((R, Hq), float("nan"), dtype=torch.float32, device="cuda") if with_lse else None
            q.qsa_gather_attn(qd, self.code, self.k_cache, self.v_cache, idx, wl.softmax_scale, out=out, lse=lse,
                              **kw)
            torch.cuda.synchronize()
            return out.cpu().numpy(), (lse.cpu().numpy() if with_lse else None), None, None
        P = num_splits
        o_part = torch.full((R, P, Hq, D), float("nan"), dtype=torch.float32, device="cuda")
        lse_part = torch.full((R, P, Hq), float("nan"), dtype=torch.float32, device="cuda")
        q.qsa_gather_attn(qd, self.code, self.k_cache, self.v_cache, idx, wl.softmax_scale, num_splits=P,
                          o_part=o_part, lse_part=lse_part, **kw)
        out = torch.full((R, Hq, D), float("nan"), dtype=torch.float32, device="cuda")
        lse = torch.full((R, Hq), float("nan"), dtype=torch.float32, device="cuda")
        q.qsa_splitk_merge(o_part, lse_part, out, lse,
                           v_scale_post=float(self.v_scale_layer) if self.fmt == "e4m3" else 1.0)
        torch.cuda.synchronize()
        return out.cpu().numpy(), lse.cpu().numpy(), o_part.cpu().numpy(), lse_part.cpu().numpy()


def _calibrated_scale_f16(x: torch.Tensor) -> float:
    import quantized_kv_cache_write_gb300 as q
    hist = torch.zeros(q.CALIB_BINS, dtype=torch.int64, device="cuda")
    rec = torch.zeros(8, dtype=torch.int64, device="cuda")
    q.qkv_calib_histogram(x.contiguous(), hist)
    q.qkv_calib_stats(hist, rec, 0.0, dtype=torch.float16)
    return q.decode_calib_stats(rec)["scale"]


class OraclePool:
    """The same slot pool written and dequantised by the CPU oracle (fp64)."""

    def __init__(self, wl, fmt: str):
        S = wl.num_slots
        self.fmt = fmt
        self.act = dt = wl.act_dtype
        self.k_scale_layer = self.v_scale_layer = None
        if fmt in ("bf16", "f16"):
            kc, vc = oq.write_bf16(wl.k_tokens, wl.v_tokens, wl.slot_mapping, S)
            widen = oatt.f16_pool_fp64 if fmt == "f16" else oatt.bf16_pool_fp64
            self.K, self.V = widen(kc), widen(vc)
            self.Vpart = self.V
            self.bytes = (kc, vc)
        elif fmt == "int8_side":
            kc, vc, ks, vs = oq.write_int8(wl.k_tokens, wl.v_tokens, wl.slot_mapping, S, "side", dtype=dt)
            self.K, self.V = oatt.int8_side_pool_fp64(kc, ks), oatt.int8_side_pool_fp64(vc, vs)
            self.Vpart = self.V
            self.bytes = (kc, vc, ks, vs)
        elif fmt == "int8_inline":
            kr, vr = oq.write_int8(wl.k_tokens, wl.v_tokens, wl.slot_mapping, S, "inline", dtype=dt)
            self.K, self.V = oatt.int8_inline_pool_fp64(kr), oatt.int8_inline_pool_fp64(vr)
            self.Vpart = self.V
            self.bytes = (kr, vr)
        elif fmt == "e4m3":
            ks = oq.e4m3_calibrated_scale(wl.k_tokens, dtype=dt)
            vs = oq.e4m3_calibrated_scale(wl.v_tokens, dtype=dt)
            self.k_scale_layer, self.v_scale_layer = ks, vs
            kc, vc = oq.write_e4m3(wl.k_tokens, wl.v_tokens, wl.slot_mapping, S, ks, vs, dtype=dt)
            self.K, self.V = oatt.e4m3_pool_fp64(kc, ks), oatt.e4m3_pool_fp64(vc, vs)
            self.Vpart = oatt.e4m3_pool_fp64(vc, vs, apply_scale=False)  # split partials: no V scale
            self.bytes = (kc, vc)
        else:
            raise ValueError(fmt)

    def attend(self, wl, rows=None):
        return oatt.gather_attention(wl.q, self.K, self.V, wl.topk, wl.softmax_scale, rows=rows, q_dtype=self.act)

    def attend_splits(self, wl, P, rows=None):
        return oatt.gather_attention_splits(wl.q, self.K, self.Vpart, wl.topk, wl.softmax_scale, P, rows=rows,
                                            q_dtype=self.act)
