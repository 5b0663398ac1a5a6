"""Thin Python binding of libqkv.so (quantize-on-write KV cache + top-k gather decode, sm_103a).

Argument marshalling only: every function takes torch tensors that already live on the GPU,
passes their device pointers, sizes and the current CUDA stream to the C entry point of
the same name declared in include/qkv.h, and raises QKVError on a non-OK status. All
arithmetic runs in the library's CUDA kernels; there is no fallback path. Importing this
package fails loudly if libqkv.so has not been built
(``python quantized_kv_cache_write_gb300/build.py``).
"""

from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libqkv.so")

QKV_OK, QKV_ERR_ARG, QKV_ERR_SCALE, QKV_ERR_UNSUPPORTED, QKV_ERR_ALIGN, QKV_ERR_CUDA = range(6)
QKV_BF16, QKV_INT8_SIDE, QKV_INT8_INLINE, QKV_E4M3, QKV_F16 = range(5)
QKV_DEV_BAD_SLOT = 1
QKV_DEV_BAD_INDEX = 2
QKV_DEV_TIMEOUT = 4
QSA_ENGINE_DEFAULT, QSA_ENGINE_TCGEN05, QSA_ENGINE_PERSISTENT = 0, 1, 2
HEAD_DIM = 256
FORMATS = {"bf16": QKV_BF16, "int8_side": QKV_INT8_SIDE, "int8_inline": QKV_INT8_INLINE, "e4m3": QKV_E4M3,
           "f16": QKV_F16}

if not os.path.exists(LIB_PATH):
    raise ImportError(f"{LIB_PATH} is missing: build it with `python quantized_kv_cache_write_gb300/build.py`")

lib = ctypes.CDLL(LIB_PATH)

_p, _i64, _i32, _f32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float
_SIGS = {
    "qkv_write_int8": [_p, _p, _i64, _i32, _i32, _i64, _p, _i32, _p, _p, _p, _p, _i64, _p, _p],
    "qkv_write_e4m3": [_p, _p, _i64, _i32, _i32, _i64, _p, _p, _p, _f32, _f32, _i64, _p, _p],
    "qkv_write_int8_f16": [_p, _p, _i64, _i32, _i32, _i64, _p, _i32, _p, _p, _p, _p, _i64, _p, _p],
    "qkv_write_e4m3_f16": [_p, _p, _i64, _i32, _i32, _i64, _p, _p, _p, _f32, _f32, _i64, _p, _p],
    "qkv_e4m3_calibrate": [_p, _i64, _p, _p, _p],
    "qkv_calib_histogram": [_p, _i64, _p, _p],
    "qkv_calib_stats": [_p, _f32, _p, _p],
    "qkv_calib_stats_f16": [_p, _f32, _p, _p],
    "qsa_gather_attn": [_p, _i64, _i32, _i32, _i32, _i32, _p, _p, _p, _p, _f32, _f32, _i64, _p, _i32, _f32,
                        _i32, _p, _p, _p, _p, _p, _p],
    "qsa_splitk_merge": [_p, _p, _i64, _i32, _i32, _i32, _f32, _p, _p, _p],
    "qsa_suggest_num_splits": [_i32, _i64, _i32, _i32, _i32, ctypes.POINTER(ctypes.c_int)],
    "qsa_gather_attn_splitk_noalloc": [_p, _i64, _i32, _i32, _i32, _i32, _p, _p, _p, _p, _f32, _f32, _i64, _p,
                                       _i32, _f32, _i32, _p, _p, _p, _p],
    "qsa_gather_attn_varlen": [_p, _i64, _i32, _i32, _i32, _i32, _p, _p, _p, _p, _f32, _f32, _i64, _p, _i32, _p,
                               _f32, _i32, _p, _p, _p, _p, _p, _p],
    "qsa_gather_attn_f16": [_p, _i64, _i32, _i32, _i32, _i32, _p, _p, _p, _p, _f32, _f32, _i64, _p, _i32, _f32,
                            _i32, _p, _p, _p, _p, _p, _p],
    "qsa_gather_attn_splitk_fused": [_p, _i64, _i32, _i32, _i32, _i32, _p, _p, _p, _p, _f32, _f32, _i64, _p, _i32,
                                     _f32, _i32, _p, _p, _p, _p, _p, _p, _p],
    "qsa_gather_attn_paged": [_p, _i64, _i32, _i32, _i32, _i32, _p, _p, _p, _p, _f32, _f32, _i64, _p, _i64, _i32,
                              _i32, _p, _p, _i32, _f32, _i32, _p, _p, _p, _p, _p, _p],
}
for _name, _args in _SIGS.items():
    _fn = getattr(lib, _name)
    _fn.argtypes = _args
    _fn.restype = ctypes.c_int
lib.qkv_status_str.argtypes = [ctypes.c_int]
lib.qkv_status_str.restype = ctypes.c_char_p


class GatherDesc(ctypes.Structure):
    """qsa_gather_desc of include/qkv.h, field for field."""
    _fields_ = [("size", ctypes.c_size_t), ("q", _p), ("q_fp16", _i32), ("rows", _i64), ("num_q_heads", _i32),
                ("num_kv_heads", _i32), ("head_dim", _i32), ("fmt", _i32), ("k_cache", _p), ("v_cache", _p),
                ("k_scale_tok", _p), ("v_scale_tok", _p), ("k_scale_layer", _f32), ("v_scale_layer", _f32),
                ("num_slots", _i64), ("topk_idx", _p), ("topk", _i32), ("softmax_scale", _f32),
                ("num_splits", _i32), ("out", _p), ("lse", _p), ("o_part", _p), ("lse_part", _p),
                ("dev_status", _p), ("topk_len", _p), ("block_table", _p), ("num_seqs", _i64),
                ("max_blocks", _i32), ("block_size", _i32), ("row_seq", _p), ("counters", _p),
                ("engine", _i32), ("sched", _p), ("shard", _i32), ("slot_lo", _i64)]


lib.qsa_gather_attn_ex.argtypes = [ctypes.POINTER(GatherDesc), _p]
lib.qsa_gather_attn_ex.restype = ctypes.c_int


class WriteDesc(ctypes.Structure):
    """qkv_write_desc of include/qkv.h, field for field."""
    _fields_ = [("size", ctypes.c_size_t), ("fmt", _i32), ("act_fp16", _i32), ("k", _p), ("v", _p),
                ("num_tokens", _i64), ("num_kv_heads", _i32), ("head_dim", _i32), ("token_stride", _i64),
                ("slot_mapping", _p), ("token_seq", _p), ("token_pos", _p), ("block_table", _p),
                ("num_seqs", _i64), ("max_blocks", _i32), ("block_size", _i32), ("k_cache", _p), ("v_cache", _p),
                ("k_scale", _p), ("v_scale", _p), ("k_scale_layer", _f32), ("v_scale_layer", _f32),
                ("num_slots", _i64), ("dev_status", _p)]


lib.qkv_write_ex.argtypes = [ctypes.POINTER(WriteDesc), _p]
lib.qkv_write_ex.restype = ctypes.c_int


class QKVError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn}: {lib.qkv_status_str(status).decode()} (status {status})")


def status_str(status: int) -> str:
    return lib.qkv_status_str(status).decode()


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(fn: str, status: int):
    if status != QKV_OK:
        raise QKVError(fn, status)


_ACT16 = (torch.bfloat16, torch.float16)


def _tokens(k: torch.Tensor, v: torch.Tensor):
    """[T, Hkv, D] views sharing one token stride; heads and dims contiguous. (The stride of a
    dimension of size 1 is never used, so it may be anything.)"""
    if k.dim() != 3 or k.shape != v.shape or k.dtype not in _ACT16 or v.dtype != k.dtype:
        raise ValueError("k and v must be bf16 (or both fp16) [num_tokens, num_kv_heads, head_dim] of equal shape")
    T, H, D = k.shape

    def heads_contiguous(t):
        return (D == 1 or t.stride(2) == 1) and (H == 1 or t.stride(1) == D)

    if not (heads_contiguous(k) and heads_contiguous(v)) or (T > 1 and k.stride(0) != v.stride(0)):
        raise ValueError("k and v need contiguous heads and one shared token stride")
    return T, H, D, (k.stride(0) if T > 1 else H * D)


def qkv_write_int8(k, v, slot_mapping, k_cache, v_cache, k_scale=None, v_scale=None, *,
                   layout: int = QKV_INT8_SIDE, dev_status=None, stream=None):
    """int8 per-(token, head) quantize-on-write (side scales or inline 260 B records); bf16 or fp16 tokens."""
    T, H, D, stride = _tokens(k, v)
    _need("slot_mapping", slot_mapping, _I64, T)
    _need("k_scale", k_scale, _F32)
    _need("v_scale", v_scale, _F32)
    _need("dev_status", dev_status, _WORD)
    name = "qkv_write_int8_f16" if k.dtype == torch.float16 else "qkv_write_int8"
    st = getattr(lib, name)(_ptr(k), _ptr(v), T, H, D, stride, _ptr(slot_mapping), layout, _ptr(k_cache),
                            _ptr(v_cache), _ptr(k_scale), _ptr(v_scale), k_cache.shape[0], _ptr(dev_status),
                            _stream(stream))
    _check(name, st)


def qkv_write_e4m3(k, v, slot_mapping, k_cache, v_cache, k_scale: float, v_scale: float, *,
                   dev_status=None, stream=None):
    """FP8 E4M3 quantize-on-write with calibrated per-layer scales; bf16 or fp16 tokens."""
    T, H, D, stride = _tokens(k, v)
    _need("slot_mapping", slot_mapping, _I64, T)
    _need("dev_status", dev_status, _WORD)
    name = "qkv_write_e4m3_f16" if k.dtype == torch.float16 else "qkv_write_e4m3"
    st = getattr(lib, name)(_ptr(k), _ptr(v), T, H, D, stride, _ptr(slot_mapping), _ptr(k_cache), _ptr(v_cache),
                            float(k_scale), float(v_scale), k_cache.shape[0], _ptr(dev_status), _stream(stream))
    _check(name, st)


def qkv_write_ex(k, v, fmt: int, k_cache, v_cache, *, slot_mapping=None, token_seq=None, token_pos=None,
                 block_table=None, block_size: int = 1, k_scale=None, v_scale=None, k_scale_layer: float = 1.0,
                 v_scale_layer: float = 1.0, dev_status=None, stream=None):
    """Any write through one descriptor (see qkv_write_ex in qkv.h): int8 side / inline or E4M3,
    bf16 or fp16 tokens, slot ids (slot_mapping) or a paged pool (token_seq, token_pos int32
    [T]; block_table int32 [num_seqs, max_blocks]; block_size)."""
    T, H, D, stride = _tokens(k, v)
    d = WriteDesc()
    d.size = ctypes.sizeof(WriteDesc)
    d.fmt, d.act_fp16 = int(fmt), int(k.dtype == torch.float16)
    d.k, d.v, d.num_tokens, d.num_kv_heads, d.head_dim, d.token_stride = _ptr(k), _ptr(v), T, H, D, stride
    d.slot_mapping, d.token_seq, d.token_pos = _ptr(slot_mapping), _ptr(token_seq), _ptr(token_pos)
    d.block_table = _ptr(block_table)
    if block_table is not None:
        if block_table.dim() != 2:
            raise ValueError("block_table must be [num_seqs, max_blocks]")
        d.num_seqs, d.max_blocks, d.block_size = block_table.shape[0], block_table.shape[1], int(block_size)
    _need("slot_mapping", slot_mapping, _I64, T)
    _need("token_seq", token_seq, _I32, T)
    _need("token_pos", token_pos, _I32, T)
    _need("block_table", block_table, _I32)
    _need("k_scale", k_scale, _F32)
    _need("v_scale", v_scale, _F32)
    _need("dev_status", dev_status, _WORD)
    d.k_cache, d.v_cache, d.k_scale, d.v_scale = _ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale)
    d.k_scale_layer, d.v_scale_layer = float(k_scale_layer), float(v_scale_layer)
    d.num_slots, d.dev_status = k_cache.shape[0], _ptr(dev_status)
    st = lib.qkv_write_ex(ctypes.byref(d), _stream(stream))
    _check("qkv_write_ex", st)


def qkv_e4m3_calibrate(x, amax_bits, scale_out, *, stream=None):
    """Device amax/448 over a bf16 tensor; result in scale_out[0] (fp32)."""
    st = lib.qkv_e4m3_calibrate(_ptr(x), x.numel(), _ptr(amax_bits), _ptr(scale_out), _stream(stream))
    _check("qkv_e4m3_calibrate", st)


CALIB_BINS = 32768  # QKV_CALIB_BINS in include/qkv.h
CALIB_STATS_BYTES = 64  # sizeof(qkv_calib_summary): six uint64 counts, then four fp32 values
_CALIB_COUNTS = ("count", "zeros", "nonfinite", "below_subnormal", "subnormal", "saturated")
_CALIB_VALUES = ("amax", "p99_9", "p99_99", "scale")


def qkv_calib_histogram(x, hist, *, stream=None):
    """Add the bf16 magnitude counts of x (any shape, contiguous) to hist (int64 [32768], device)."""
    if x.dtype not in _ACT16 or not x.is_contiguous():
        raise ValueError("x must be a contiguous bf16 or fp16 tensor")
    if hist.numel() != CALIB_BINS or hist.element_size() != 8:
        raise ValueError(f"hist must hold {CALIB_BINS} 64-bit counts")
    st = lib.qkv_calib_histogram(_ptr(x), x.numel(), _ptr(hist), _stream(stream))
    _check("qkv_calib_histogram", st)


def qkv_calib_stats(hist, stats, scale: float = 0.0, *, dtype=torch.bfloat16, stream=None):
    """Statistics of a histogram into stats (a 64-byte device buffer, e.g. int64 [8]).

    scale 0 uses the calibrated amax / 448; dtype is the type the histogram counted (bf16 or
    fp16); read the record with decode_calib_stats.
    """
    if stats.numel() * stats.element_size() < CALIB_STATS_BYTES:
        raise ValueError(f"stats must hold {CALIB_STATS_BYTES} bytes")
    if dtype not in _ACT16:
        raise ValueError("dtype must be torch.bfloat16 or torch.float16")
    name = "qkv_calib_stats_f16" if dtype == torch.float16 else "qkv_calib_stats"
    st = getattr(lib, name)(_ptr(hist), float(scale), _ptr(stats), _stream(stream))
    _check(name, st)


def decode_calib_stats(stats) -> dict:
    """The qkv_calib_summary record in a device or host buffer, as a dict (copies to the host)."""
    raw = stats.detach().contiguous().view(torch.uint8)[:CALIB_STATS_BYTES].cpu()
    counts = raw[:48].view(torch.int64).tolist()
    values = raw[48:64].view(torch.float32).tolist()
    return {**dict(zip(_CALIB_COUNTS, counts)), **dict(zip(_CALIB_VALUES, values))}


def _expect_shape(name: str, t, shape):
    if t is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")


_I32 = (torch.int32,)
_I64 = (torch.int64,)
_F32 = (torch.float32,)
_WORD = (torch.int32, torch.uint32)


def _need(name: str, t, dtypes, numel: Optional[int] = None):
    """A tensor the kernels read or write by raw pointer: its dtype, contiguity and size."""
    if t is None:
        return
    if t.dtype not in dtypes:
        raise ValueError(f"{name} must be {' or '.join(str(d).replace('torch.', '') for d in dtypes)}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if numel is not None and t.numel() != numel:
        raise ValueError(f"{name} must hold {numel} elements, got {t.numel()}")


def _check_gather_shapes(q, topk_idx, num_splits, out, lse, o_part=None, lse_part=None):
    """The kernels index every buffer by q's row count: the others must agree with it."""
    R, Hq, D = q.shape
    if topk_idx is not None and (topk_idx.dim() != 2 or topk_idx.shape[0] != R):
        raise ValueError(f"topk_idx must be [{R}, k], got {tuple(topk_idx.shape)}")
    _need("topk_idx", topk_idx, _I32)
    _expect_shape("out", out, (R, Hq, D))
    _expect_shape("lse", lse, (R, Hq))
    _expect_shape("o_part", o_part, (R, num_splits, Hq, D))
    _expect_shape("lse_part", lse_part, (R, num_splits, Hq))
    for name, t in (("out", out), ("lse", lse), ("o_part", o_part), ("lse_part", lse_part)):
        _need(name, t, _F32)


def _check_gather_aux(k_scale_tok, v_scale_tok, dev_status, counters=None, row_seq=None, block_table=None,
                      topk_len=None, rows=None):
    _need("k_scale_tok", k_scale_tok, _F32)
    _need("v_scale_tok", v_scale_tok, _F32)
    _need("dev_status", dev_status, _WORD)
    _need("counters", counters, _WORD)
    _need("row_seq", row_seq, _I32, rows)
    _need("block_table", block_table, _I32)
    _need("topk_len", topk_len, _I32, rows)


def qsa_gather_attn(q, fmt: int, k_cache, v_cache, topk_idx, softmax_scale: float, *, num_kv_heads: int = 1,
                    num_slots: Optional[int] = None, k_scale_tok=None, v_scale_tok=None,
                    k_scale_layer: float = 1.0, v_scale_layer: float = 1.0, num_splits: int = 1, out=None,
                    lse=None, o_part=None, lse_part=None, dev_status=None, stream=None):
    """Top-k gather decode attention. q bf16 (or fp16: qsa_gather_attn_f16) [R, Hq, D]; topk_idx int32 [R, k]."""
    _check_gather_shapes(q, topk_idx, num_splits, out, lse, o_part, lse_part)
    _check_gather_aux(k_scale_tok, v_scale_tok, dev_status)
    R, Hq, D = q.shape
    S = k_cache.shape[0] if num_slots is None else num_slots
    topk = topk_idx.shape[1] if topk_idx is not None else 0
    name = "qsa_gather_attn_f16" if q.dtype == torch.float16 else "qsa_gather_attn"
    st = getattr(lib, name)(_ptr(q), R, Hq, num_kv_heads, D, fmt, _ptr(k_cache), _ptr(v_cache),
                            _ptr(k_scale_tok), _ptr(v_scale_tok), float(k_scale_layer), float(v_scale_layer), S,
                            _ptr(topk_idx), topk, float(softmax_scale), num_splits, _ptr(out), _ptr(lse),
                            _ptr(o_part), _ptr(lse_part), _ptr(dev_status), _stream(stream))
    _check(name, st)


def qsa_gather_attn_varlen(q, fmt: int, k_cache, v_cache, topk_idx, topk_len, softmax_scale: float, *,
                           num_kv_heads: int = 1, num_slots: Optional[int] = None, k_scale_tok=None,
                           v_scale_tok=None, k_scale_layer: float = 1.0, v_scale_layer: float = 1.0,
                           num_splits: int = 1, out=None, lse=None, o_part=None, lse_part=None, dev_status=None,
                           stream=None):
    """Gather for rows of different lengths: row r uses topk_idx[r, :topk_len[r]] (int32 [R])."""
    _check_gather_shapes(q, topk_idx, num_splits, out, lse, o_part, lse_part)
    R, Hq, D = q.shape
    if topk_len is None or topk_len.numel() != R or topk_len.dtype != torch.int32:
        raise ValueError(f"topk_len must be int32 [{R}]")
    _check_gather_aux(k_scale_tok, v_scale_tok, dev_status, topk_len=topk_len, rows=R)
    S = k_cache.shape[0] if num_slots is None else num_slots
    topk = topk_idx.shape[1]
    st = lib.qsa_gather_attn_varlen(_ptr(q), R, Hq, num_kv_heads, D, fmt, _ptr(k_cache), _ptr(v_cache),
                                    _ptr(k_scale_tok), _ptr(v_scale_tok), float(k_scale_layer), float(v_scale_layer),
                                    S, _ptr(topk_idx), topk, _ptr(topk_len), float(softmax_scale), num_splits,
                                    _ptr(out), _ptr(lse), _ptr(o_part), _ptr(lse_part), _ptr(dev_status),
                                    _stream(stream))
    _check("qsa_gather_attn_varlen", st)


def qsa_gather_attn_ex(q, fmt: int, k_cache, v_cache, topk_idx, softmax_scale: float, *, num_kv_heads: int = 1,
                       num_slots: Optional[int] = None, k_scale_tok=None, v_scale_tok=None,
                       k_scale_layer: float = 1.0, v_scale_layer: float = 1.0, num_splits: int = 1, out=None,
                       lse=None, o_part=None, lse_part=None, dev_status=None, topk_len=None, block_table=None,
                       row_seq=None, block_size: int = 0, counters=None, engine: int = 0, sched=None,
                       slot_lo: Optional[int] = None, stream=None):
    """Any combination of the gather's options in one call (see qsa_gather_attn_ex in qkv.h).

    q bf16 or fp16 [R, Hq, D]; topk_len int32 [R] (varlen); block_table int32 [num_seqs,
    max_blocks] with row_seq int32 [R] and block_size (paged: topk_idx holds positions);
    counters [R, Hkv, ceil(G / 16)] (fused split-K merge into out / lse); engine
    QSA_ENGINE_TCGEN05 selects the tensor-memory q.K^T variant of the int8 side gather;
    QSA_ENGINE_PERSISTENT runs on a resident grid that takes work items from sched (int32 or
    uint32 [2], zero on the first call and left zero). slot_lo (not None): this pool is the
    shard of global slots [slot_lo, slot_lo + num_slots); topk_idx holds global ids and entries
    of other shards are skipped.
    """
    _check_gather_shapes(q, topk_idx, num_splits, out, lse, o_part, lse_part)
    R, Hq, D = q.shape
    if topk_len is not None and (topk_len.numel() != R or topk_len.dtype != torch.int32):
        raise ValueError(f"topk_len must be int32 [{R}]")
    if block_table is not None and (block_table.dim() != 2 or row_seq is None or row_seq.numel() != R):
        raise ValueError(f"block_table must be [num_seqs, max_blocks] with row_seq [{R}]")
    if counters is not None and counters.numel() != R * num_kv_heads * ((Hq // num_kv_heads + 15) // 16):
        raise ValueError("counters must hold rows x num_kv_heads x ceil(G / 16) entries")
    _check_gather_aux(k_scale_tok, v_scale_tok, dev_status, counters, row_seq, block_table, topk_len, R)
    _need("sched", sched, _WORD, None if sched is None else 2)
    if sched is not None and sched.device != q.device:
        raise ValueError("sched must be on the query's device")
    d = GatherDesc()
    d.size = ctypes.sizeof(GatherDesc)
    d.q, d.q_fp16, d.rows, d.num_q_heads, d.num_kv_heads, d.head_dim = _ptr(q), int(q.dtype == torch.float16), R, Hq, \
        num_kv_heads, D
    d.fmt, d.k_cache, d.v_cache = fmt, _ptr(k_cache), _ptr(v_cache)
    d.k_scale_tok, d.v_scale_tok = _ptr(k_scale_tok), _ptr(v_scale_tok)
    d.k_scale_layer, d.v_scale_layer = float(k_scale_layer), float(v_scale_layer)
    d.num_slots = k_cache.shape[0] if num_slots is None else num_slots
    d.topk_idx, d.topk, d.softmax_scale, d.num_splits = _ptr(topk_idx), topk_idx.shape[1], float(softmax_scale), \
        num_splits
    d.out, d.lse, d.o_part, d.lse_part, d.dev_status = _ptr(out), _ptr(lse), _ptr(o_part), _ptr(lse_part), \
        _ptr(dev_status)
    d.topk_len, d.counters, d.engine, d.sched = _ptr(topk_len), _ptr(counters), int(engine), _ptr(sched)
    d.shard, d.slot_lo = (0, 0) if slot_lo is None else (1, int(slot_lo))
    if block_table is not None:
        d.block_table, d.num_seqs, d.max_blocks, d.block_size = _ptr(block_table), block_table.shape[0], \
            block_table.shape[1], int(block_size)
        d.row_seq = _ptr(row_seq)
    st = lib.qsa_gather_attn_ex(ctypes.byref(d), _stream(stream))
    _check("qsa_gather_attn_ex", st)


def qsa_gather_attn_paged(q, fmt: int, k_cache, v_cache, block_table, row_seq, topk_pos, block_size: int,
                          softmax_scale: float, *, num_kv_heads: int = 1, num_slots: Optional[int] = None,
                          k_scale_tok=None, v_scale_tok=None, k_scale_layer: float = 1.0,
                          v_scale_layer: float = 1.0, num_splits: int = 1, out=None, lse=None, o_part=None,
                          lse_part=None, dev_status=None, stream=None):
    """Top-k gather decode attention over a paged pool.

    block_table int32 [num_seqs, max_blocks]; row_seq int32 [R]; topk_pos int32 [R, k] logical
    positions (-1 padding); slot = block_table[seq, pos // block_size] * block_size + pos % block_size.
    """
    _check_gather_shapes(q, topk_pos, num_splits, out, lse, o_part, lse_part)
    R, Hq, D = q.shape
    if block_table.dim() != 2 or row_seq.dim() != 1 or row_seq.shape[0] != R:
        raise ValueError(f"block_table must be [num_seqs, max_blocks] and row_seq [{R}]")
    _check_gather_aux(k_scale_tok, v_scale_tok, dev_status, row_seq=row_seq, block_table=block_table, rows=R)
    S = k_cache.shape[0] if num_slots is None else num_slots
    topk = topk_pos.shape[1] if topk_pos is not None else 0
    st = lib.qsa_gather_attn_paged(_ptr(q), R, Hq, num_kv_heads, D, fmt, _ptr(k_cache), _ptr(v_cache),
                                   _ptr(k_scale_tok), _ptr(v_scale_tok), float(k_scale_layer),
                                   float(v_scale_layer), S, _ptr(block_table), block_table.shape[0],
                                   block_table.shape[1], int(block_size), _ptr(row_seq), _ptr(topk_pos), topk,
                                   float(softmax_scale), num_splits, _ptr(out), _ptr(lse), _ptr(o_part),
                                   _ptr(lse_part), _ptr(dev_status), _stream(stream))
    _check("qsa_gather_attn_paged", st)


def qsa_gather_attn_splitk_fused(q, fmt: int, k_cache, v_cache, topk_idx, softmax_scale: float, *, num_splits: int,
                                 out, o_part, lse_part, counters, lse=None, num_kv_heads: int = 1,
                                 num_slots: Optional[int] = None, k_scale_tok=None, v_scale_tok=None,
                                 k_scale_layer: float = 1.0, v_scale_layer: float = 1.0, dev_status=None,
                                 stream=None):
    """Split-K gather with the merge fused into the same launch (the last split CTA merges).

    counters: int32/uint32 [R, num_kv_heads, ceil(G / 16)], all zero before the first call and
    left zero (G = num_q_heads / num_kv_heads).
    """
    _check_gather_shapes(q, topk_idx, num_splits, out, lse, o_part, lse_part)
    R, Hq, D = q.shape
    chunks = (Hq // num_kv_heads + 15) // 16
    if counters is not None and counters.numel() != R * num_kv_heads * chunks:
        raise ValueError(f"counters must hold {R} x {num_kv_heads} x {chunks} entries, got {counters.numel()}")
    _check_gather_aux(k_scale_tok, v_scale_tok, dev_status, counters)
    S = k_cache.shape[0] if num_slots is None else num_slots
    topk = topk_idx.shape[1] if topk_idx is not None else 0
    st = lib.qsa_gather_attn_splitk_fused(_ptr(q), R, Hq, num_kv_heads, D, fmt, _ptr(k_cache), _ptr(v_cache),
                                          _ptr(k_scale_tok), _ptr(v_scale_tok), float(k_scale_layer),
                                          float(v_scale_layer), S, _ptr(topk_idx), topk, float(softmax_scale),
                                          num_splits, _ptr(out), _ptr(lse), _ptr(o_part), _ptr(lse_part),
                                          _ptr(counters), _ptr(dev_status), _stream(stream))
    _check("qsa_gather_attn_splitk_fused", st)


def qsa_suggest_num_splits(fmt: int, rows: int, num_q_heads: int, num_kv_heads: int, topk: int) -> int:
    """Split count that fills one wave of resident CTAs on the current device."""
    out = ctypes.c_int(0)
    st = lib.qsa_suggest_num_splits(fmt, rows, num_q_heads, num_kv_heads, topk, ctypes.byref(out))
    _check("qsa_suggest_num_splits", st)
    return out.value


def qsa_splitk_merge(o_part, lse_part, out, lse=None, *, v_scale_post: float = 1.0, stream=None):
    """Merge split-K partials o_part [R, P, Hq, D], lse_part [R, P, Hq] into out [R, Hq, D]."""
    R, P, Hq, D = o_part.shape
    _expect_shape("lse_part", lse_part, (R, P, Hq))
    _expect_shape("out", out, (R, Hq, D))
    _expect_shape("lse", lse, (R, Hq))
    for name, t in (("o_part", o_part), ("lse_part", lse_part), ("out", out), ("lse", lse)):
        _need(name, t, _F32)
    st = lib.qsa_splitk_merge(_ptr(o_part), _ptr(lse_part), R, Hq, D, P, float(v_scale_post), _ptr(out), _ptr(lse),
                              _stream(stream))
    _check("qsa_splitk_merge", st)


NOALLOC_SCRATCH_BYTES = 16 * 1024 * 1024  # QKV_NOALLOC_SCRATCH_BYTES in include/qkv.h


def noalloc_scratch_bytes(rows: int, num_splits: int, num_q_heads: int, head_dim: int = HEAD_DIM) -> int:
    """Bytes of the library's static scratch that a split call of this size needs."""
    parts = rows * num_splits * num_q_heads
    return ((parts * head_dim * 4 + 255) // 256) * 256 + parts * 4


def qsa_gather_attn_splitk_noalloc(q, fmt: int, k_cache, v_cache, topk_idx, softmax_scale: float, *,
                                   num_splits: int, out, lse=None, num_kv_heads: int = 1,
                                   num_slots: Optional[int] = None, k_scale_tok=None, v_scale_tok=None,
                                   k_scale_layer: float = 1.0, v_scale_layer: float = 1.0, dev_status=None,
                                   stream=None):
    """Split-K gather + merge with the partials in the library's static device scratch.

    For callers that may not allocate device memory: only inputs and outputs are passed.
    Calls share one scratch array per GPU, so calls that overlap on the GPU race.
    """
    _check_gather_shapes(q, topk_idx, num_splits, out, lse)
    _check_gather_aux(k_scale_tok, v_scale_tok, dev_status)
    R, Hq, D = q.shape
    if num_splits > 1 and noalloc_scratch_bytes(R, num_splits, Hq, D) > NOALLOC_SCRATCH_BYTES:
        raise ValueError(f"{R} rows x {num_splits} splits x {Hq} heads needs "
                         f"{noalloc_scratch_bytes(R, num_splits, Hq, D)} bytes of partials, more than the "
                         f"{NOALLOC_SCRATCH_BYTES}-byte static scratch of qsa_gather_attn_splitk_noalloc")
    S = k_cache.shape[0] if num_slots is None else num_slots
    topk = topk_idx.shape[1] if topk_idx is not None else 0
    st = lib.qsa_gather_attn_splitk_noalloc(_ptr(q), R, Hq, num_kv_heads, D, fmt, _ptr(k_cache), _ptr(v_cache),
                                            _ptr(k_scale_tok), _ptr(v_scale_tok), float(k_scale_layer),
                                            float(v_scale_layer), S, _ptr(topk_idx), topk, float(softmax_scale),
                                            num_splits, _ptr(out), _ptr(lse), _ptr(dev_status), _stream(stream))
    _check("qsa_gather_attn_splitk_noalloc", st)
