"""The C ABI without a GPU: libqkv.so builds, exports every function include/qkv.h declares,
and its host-side validation rejects bad calls before any CUDA work (these calls return
before the first CUDA API call, so they are safe on a machine with no GPU).

The fail-closed scale gate follows "[Model][SM70][FP8] Add calibrated E4M3 QSA KV cache"
§Non-obvious design decisions: a missing (-1.0 sentinel), non-finite or non-positive
per-layer scale is an error; 1.0 is a legal value.
"""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "qkv.h")


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    path = __graft_entry__._builder().build()
    import quantized_kv_cache_write_gb300 as q
    assert q.LIB_PATH == path
    return q


def _declared():
    text = open(HEADER).read()
    return re.findall(r"^\s*(?:qkv_status|const char\*)\s+(\w+)\s*\(", text, flags=re.M)


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert {"qkv_write_int8", "qkv_write_e4m3", "qsa_gather_attn", "qsa_splitk_merge", "qkv_status_str"} <= set(names)
    raw = ctypes.CDLL(lib.LIB_PATH)
    for n in names:
        assert hasattr(raw, n), n


def test_status_strings(lib):
    for s in range(6):
        assert lib.status_str(s)
    assert lib.status_str(99) == "unknown status"


FAKE = 0x10000  # a 64 KiB-aligned fake device address: never dereferenced, the calls fail first


def _gather(lib, **over):
    a = dict(q=FAKE, rows=4, hq=16, hkv=1, d=256, fmt=lib.QKV_INT8_SIDE, kc=FAKE, vc=FAKE, ks=FAKE, vs=FAKE,
             ksl=1.0, vsl=1.0, S=100, idx=FAKE, topk=8, sm=0.0625, P=1, out=FAKE, lse=None, op=None, lp=None)
    a.update(over)
    return lib.lib.qsa_gather_attn(a["q"], a["rows"], a["hq"], a["hkv"], a["d"], a["fmt"], a["kc"], a["vc"], a["ks"],
                                   a["vs"], a["ksl"], a["vsl"], a["S"], a["idx"], a["topk"], a["sm"], a["P"],
                                   a["out"], a["lse"], a["op"], a["lp"], None, None)


def test_gather_host_validation(lib):
    E = lib
    assert _gather(lib, d=64) == E.QKV_ERR_UNSUPPORTED
    assert _gather(lib, d=128, rows=0) == E.QKV_OK  # 128-wide heads are supported
    assert _gather(lib, hq=258, hkv=2) == E.QKV_ERR_UNSUPPORTED  # group 129
    assert _gather(lib, hq=256, hkv=2, rows=0) == E.QKV_OK  # group 128 is supported
    assert _gather(lib, hq=15, hkv=2) == E.QKV_ERR_ARG
    assert _gather(lib, fmt=7) == E.QKV_ERR_ARG
    assert _gather(lib, ks=None) == E.QKV_ERR_ARG  # side format needs per-slot scales
    assert _gather(lib, fmt=E.QKV_E4M3) == E.QKV_ERR_ARG  # ... and the others must not get them
    assert _gather(lib, P=2) == E.QKV_ERR_ARG  # split needs partial buffers, not out
    assert _gather(lib, P=0) == E.QKV_ERR_ARG
    assert _gather(lib, rows=-1) == E.QKV_ERR_ARG
    assert _gather(lib, sm=float("nan")) == E.QKV_ERR_ARG
    assert _gather(lib, q=FAKE + 8) == E.QKV_ERR_ALIGN
    assert _gather(lib, out=FAKE + 4) == E.QKV_ERR_ALIGN
    assert _gather(lib, rows=0) == E.QKV_OK  # nothing to do, nothing launched


@pytest.mark.parametrize("bad", [-1.0, 0.0, float("nan"), float("inf"), -0.0])
def test_e4m3_scale_gate_fails_closed(lib, bad):
    E = lib
    kw = dict(fmt=E.QKV_E4M3, ks=None, vs=None)
    assert _gather(lib, ksl=bad, **kw) == E.QKV_ERR_SCALE
    assert _gather(lib, vsl=bad, **kw) == E.QKV_ERR_SCALE
    st = lib.lib.qkv_write_e4m3(FAKE, FAKE, 3, 1, 256, 256, FAKE, FAKE, FAKE, bad, 1.0, 10, None, None)
    assert st == E.QKV_ERR_SCALE


def test_unit_scale_is_legal(lib):
    # 1.0 passes the gate; rows=0 keeps the call from launching anything
    assert _gather(lib, fmt=lib.QKV_E4M3, ks=None, vs=None, ksl=1.0, vsl=1.0, rows=0) == lib.QKV_OK


def test_write_host_validation(lib):
    E, L = lib, lib.lib
    w8 = lambda **o: L.qkv_write_int8(o.get("k", FAKE), FAKE, o.get("T", 3), 1, o.get("d", 256), o.get("ts", 256),
                                      FAKE, o.get("layout", E.QKV_INT8_SIDE), FAKE, FAKE, o.get("ks", FAKE),
                                      o.get("vs", FAKE), 10, None, None)
    assert w8(d=64) == E.QKV_ERR_UNSUPPORTED
    assert w8(ts=100) == E.QKV_ERR_ARG  # stride below one token
    assert w8(ts=260) == E.QKV_ERR_ALIGN
    assert w8(k=FAKE + 2) == E.QKV_ERR_ALIGN
    assert w8(layout=E.QKV_E4M3) == E.QKV_ERR_ARG
    assert w8(layout=E.QKV_INT8_INLINE) == E.QKV_ERR_ARG  # inline must not get scale pointers
    assert w8(ks=None) == E.QKV_ERR_ARG
    assert w8(T=-1) == E.QKV_ERR_ARG
    assert w8(T=(1 << 32) + 1) == E.QKV_ERR_ARG  # more head rows than one launch's grid holds
    assert w8(T=0) == E.QKV_OK


def test_merge_and_calibrate_host_validation(lib):
    E, L = lib, lib.lib
    assert L.qsa_splitk_merge(FAKE, FAKE, 2, 16, 192, 4, 1.0, FAKE, None, None) == E.QKV_ERR_UNSUPPORTED
    assert L.qsa_splitk_merge(FAKE, FAKE, 1 << 29, 16, 256, 4, 1.0, FAKE, None, None) == E.QKV_ERR_ARG
    assert L.qsa_splitk_merge(FAKE, FAKE, 2, 16, 256, 0, 1.0, FAKE, None, None) == E.QKV_ERR_ARG
    assert L.qsa_splitk_merge(FAKE, FAKE, 2, 16, 256, 4, float("inf"), FAKE, None, None) == E.QKV_ERR_ARG
    assert L.qsa_splitk_merge(FAKE + 4, FAKE, 2, 16, 256, 4, 1.0, FAKE, None, None) == E.QKV_ERR_ALIGN
    assert L.qsa_splitk_merge(FAKE, FAKE, 0, 16, 256, 4, 1.0, FAKE, None, None) == E.QKV_OK
    assert L.qkv_e4m3_calibrate(FAKE, -1, FAKE, FAKE, None) == E.QKV_ERR_ARG
    assert L.qkv_e4m3_calibrate(FAKE + 2, 10, FAKE, FAKE, None) == E.QKV_ERR_ALIGN


def test_binding_rejects_buffers_that_disagree_with_q(lib):
    """The kernels index every buffer by q's row count; the binding refuses a mismatch
    before any call, so a short topk_idx or out can never be read or written past its end."""
    import torch
    q = torch.zeros((4, 16, 256), dtype=torch.bfloat16)
    kc = torch.zeros((8, 1, 256), dtype=torch.int8)
    idx_ok = torch.zeros((4, 5), dtype=torch.int32)
    out_ok = torch.zeros((4, 16, 256), dtype=torch.float32)
    cases = [
        dict(topk_idx=torch.zeros((3, 5), dtype=torch.int32), out=out_ok),
        dict(topk_idx=idx_ok, out=torch.zeros((3, 16, 256), dtype=torch.float32)),
        dict(topk_idx=idx_ok, out=out_ok, lse=torch.zeros((4, 8), dtype=torch.float32)),
        dict(topk_idx=idx_ok, out=None, num_splits=2, o_part=torch.zeros((4, 3, 16, 256)),
             lse_part=torch.zeros((4, 2, 16))),
    ]
    for kw in cases:
        with pytest.raises(ValueError):
            lib.qsa_gather_attn(q, lib.QKV_INT8_SIDE, kc, kc, kw.pop("topk_idx"), 0.0625, **kw)
    with pytest.raises(ValueError):
        lib.qsa_splitk_merge(torch.zeros((4, 2, 16, 256)), torch.zeros((4, 3, 16)), out_ok)
    with pytest.raises(ValueError):
        lib.qsa_gather_attn_splitk_noalloc(q, lib.QKV_INT8_SIDE, kc, kc, idx_ok, 0.0625, num_splits=2,
                                           out=torch.zeros((2, 16, 256)))


def test_token_views_ignore_the_strides_of_unit_dimensions(lib):
    """A dimension of size 1 is never stepped over, so its stride (0 for a broadcast view) does
    not matter; real mismatches are still refused."""
    import torch
    base = torch.zeros((5, 256), dtype=torch.bfloat16)
    k = base.as_strided((5, 1, 256), (256, 0, 1))
    assert lib._tokens(k, k) == (5, 1, 256, 256)
    one = base.as_strided((1, 1, 256), (0, 0, 1))
    assert lib._tokens(one, one) == (1, 1, 256, 256)
    two = torch.zeros((5, 2, 256), dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        lib._tokens(two.transpose(0, 1).contiguous().transpose(0, 1), two)  # heads not contiguous
    with pytest.raises(ValueError):
        lib._tokens(torch.zeros((5, 1, 512), dtype=torch.bfloat16)[:, :, :256], k)  # token strides differ


def test_binding_checks_raw_pointer_tensors(lib):
    """Index, scale and output tensors reach the kernels as raw pointers: the binding refuses a
    wrong dtype, a non-contiguous view or a wrong length before any call."""
    import torch
    k = torch.zeros((4, 1, 256), dtype=torch.bfloat16)
    kc = torch.zeros((8, 1, 256), dtype=torch.int8)
    sc = torch.zeros((8, 1), dtype=torch.float32)
    sm = torch.arange(4, dtype=torch.int64)
    with pytest.raises(ValueError, match="slot_mapping must be int64"):
        lib.qkv_write_int8(k, k, sm.to(torch.int32), kc, kc, sc, sc)
    with pytest.raises(ValueError, match="slot_mapping must hold 4"):
        lib.qkv_write_int8(k, k, torch.arange(5, dtype=torch.int64), kc, kc, sc, sc)
    with pytest.raises(ValueError, match="k_scale must be float32"):
        lib.qkv_write_int8(k, k, sm, kc, kc, sc.double(), sc)
    with pytest.raises(ValueError, match="dev_status"):
        lib.qkv_write_e4m3(k, k, sm, kc, kc, 1.0, 1.0, dev_status=torch.zeros(1))
    with pytest.raises(ValueError, match="token_pos must be int32"):
        lib.qkv_write_ex(k, k, lib.QKV_E4M3, kc, kc, token_seq=torch.zeros(4, dtype=torch.int32),
                         token_pos=torch.zeros(4, dtype=torch.int64), block_table=torch.zeros((2, 2), dtype=torch.int32),
                         block_size=16)
    q = torch.zeros((4, 16, 256), dtype=torch.bfloat16)
    out = torch.zeros((4, 16, 256), dtype=torch.float32)
    idx = torch.zeros((4, 6), dtype=torch.int32)
    with pytest.raises(ValueError, match="topk_idx must be int32"):
        lib.qsa_gather_attn(q, lib.QKV_INT8_SIDE, kc, kc, idx.long(), 0.0625, out=out)
    with pytest.raises(ValueError, match="topk_idx must be contiguous"):
        lib.qsa_gather_attn(q, lib.QKV_INT8_SIDE, kc, kc, torch.zeros((6, 4), dtype=torch.int32).t(), 0.0625, out=out)
    with pytest.raises(ValueError, match="out must be float32"):
        lib.qsa_gather_attn(q, lib.QKV_INT8_SIDE, kc, kc, idx, 0.0625, out=out.double())
    with pytest.raises(ValueError, match="counters"):
        lib.qsa_gather_attn_splitk_fused(q, lib.QKV_INT8_SIDE, kc, kc, idx, 0.0625, num_splits=2, out=out,
                                         o_part=torch.zeros((4, 2, 16, 256)), lse_part=torch.zeros((4, 2, 16)),
                                         counters=torch.zeros(4, dtype=torch.int64))
    with pytest.raises(ValueError, match="o_part must be float32"):
        lib.qsa_splitk_merge(torch.zeros((4, 2, 16, 256), dtype=torch.float64), torch.zeros((4, 2, 16)), out)


def _gather_paged(lib, **over):
    a = dict(q=FAKE, rows=4, hq=16, hkv=1, d=256, fmt=lib.QKV_INT8_SIDE, kc=FAKE, vc=FAKE, ks=FAKE, vs=FAKE,
             ksl=1.0, vsl=1.0, S=100, bt=FAKE, nseq=2, mb=8, bs=16, rs=FAKE, pos=FAKE, topk=8, sm=0.0625, P=1,
             out=FAKE, lse=None, op=None, lp=None)
    a.update(over)
    return lib.lib.qsa_gather_attn_paged(a["q"], a["rows"], a["hq"], a["hkv"], a["d"], a["fmt"], a["kc"], a["vc"],
                                         a["ks"], a["vs"], a["ksl"], a["vsl"], a["S"], a["bt"], a["nseq"], a["mb"],
                                         a["bs"], a["rs"], a["pos"], a["topk"], a["sm"], a["P"], a["out"], a["lse"],
                                         a["op"], a["lp"], None, None)


def test_paged_gather_host_validation(lib):
    E = lib
    assert _gather_paged(lib, bs=0) == E.QKV_ERR_ARG
    assert _gather_paged(lib, mb=0) == E.QKV_ERR_ARG
    assert _gather_paged(lib, nseq=0) == E.QKV_ERR_ARG
    assert _gather_paged(lib, mb=1 << 20, bs=1 << 12) == E.QKV_ERR_ARG  # positions would pass 2^31
    assert _gather_paged(lib, bt=None) == E.QKV_ERR_ARG
    assert _gather_paged(lib, rs=None) == E.QKV_ERR_ARG
    assert _gather_paged(lib, rs=FAKE + 2) == E.QKV_ERR_ALIGN
    assert _gather_paged(lib, d=96) == E.QKV_ERR_UNSUPPORTED  # the common checks still apply
    assert _gather_paged(lib, rows=0) == E.QKV_OK


def _gather_fused(lib, **over):
    a = dict(q=FAKE, rows=4, hq=16, hkv=1, d=256, fmt=lib.QKV_INT8_SIDE, kc=FAKE, vc=FAKE, ks=FAKE, vs=FAKE,
             ksl=1.0, vsl=1.0, S=100, idx=FAKE, topk=8, sm=0.0625, P=4, out=FAKE, lse=None, op=FAKE, lp=FAKE,
             cnt=FAKE)
    a.update(over)
    return lib.lib.qsa_gather_attn_splitk_fused(a["q"], a["rows"], a["hq"], a["hkv"], a["d"], a["fmt"], a["kc"],
                                                a["vc"], a["ks"], a["vs"], a["ksl"], a["vsl"], a["S"], a["idx"],
                                                a["topk"], a["sm"], a["P"], a["out"], a["lse"], a["op"], a["lp"],
                                                a["cnt"], None, None)


def test_fused_gather_host_validation(lib):
    E = lib
    assert _gather_fused(lib, cnt=None) == E.QKV_ERR_ARG  # a split call needs the arrival counters
    assert _gather_fused(lib, cnt=FAKE + 2) == E.QKV_ERR_ALIGN
    assert _gather_fused(lib, out=None) == E.QKV_ERR_ARG  # ... the merged output
    assert _gather_fused(lib, op=None) == E.QKV_ERR_ARG  # ... and the partial workspace
    assert _gather_fused(lib, lp=None) == E.QKV_ERR_ARG
    assert _gather_fused(lib, out=FAKE + 4) == E.QKV_ERR_ALIGN
    assert _gather_fused(lib, P=0) == E.QKV_ERR_ARG
    assert _gather_fused(lib, d=512) == E.QKV_ERR_UNSUPPORTED
    assert _gather_fused(lib, fmt=E.QKV_E4M3, ks=None, vs=None, ksl=0.0) == E.QKV_ERR_SCALE
    assert _gather_fused(lib, rows=0) == E.QKV_OK
    # unsplit: workspace and counters are neither needed nor allowed to be required
    assert _gather_fused(lib, P=1, op=None, lp=None, cnt=None, rows=0) == E.QKV_OK


def test_calibration_host_validation(lib):
    E, L = lib, lib.lib
    assert L.qkv_calib_histogram(FAKE, -1, FAKE, None) == E.QKV_ERR_ARG
    assert L.qkv_calib_histogram(FAKE, 1 << 41, FAKE, None) == E.QKV_ERR_ARG
    assert L.qkv_calib_histogram(FAKE, 10, None, None) == E.QKV_ERR_ARG
    assert L.qkv_calib_histogram(FAKE + 2, 10, FAKE, None) == E.QKV_ERR_ALIGN
    assert L.qkv_calib_histogram(FAKE, 10, FAKE + 4, None) == E.QKV_ERR_ALIGN
    assert L.qkv_calib_histogram(None, 0, FAKE, None) == E.QKV_OK  # nothing to count
    for bad in (-1.0, float("nan"), float("inf")):
        assert L.qkv_calib_stats(FAKE, bad, FAKE, None) == E.QKV_ERR_SCALE
    assert L.qkv_calib_stats(None, 0.0, FAKE, None) == E.QKV_ERR_ARG
    assert L.qkv_calib_stats(FAKE, 0.0, FAKE + 4, None) == E.QKV_ERR_ALIGN


def test_suggest_num_splits_host_validation(lib):
    import ctypes
    E, L = lib, lib.lib
    out = ctypes.c_int(0)
    assert L.qsa_suggest_num_splits(E.QKV_INT8_SIDE, 40, 16, 1, 2048, None) == E.QKV_ERR_ARG
    assert L.qsa_suggest_num_splits(E.QKV_INT8_SIDE, -1, 16, 1, 2048, ctypes.byref(out)) == E.QKV_ERR_ARG
    assert L.qsa_suggest_num_splits(E.QKV_INT8_SIDE, 40, 15, 2, 2048, ctypes.byref(out)) == E.QKV_ERR_ARG
    assert L.qsa_suggest_num_splits(E.QKV_INT8_SIDE, 40, 258, 2, 2048, ctypes.byref(out)) == E.QKV_ERR_UNSUPPORTED
    assert L.qsa_suggest_num_splits(7, 40, 16, 1, 2048, ctypes.byref(out)) == E.QKV_ERR_ARG


def test_fp16_entry_points_host_validation(lib):
    E, L = lib, lib.lib
    g16 = lambda fmt, **o: L.qsa_gather_attn_f16(FAKE, o.get("rows", 4), 16, 1, 256, fmt, FAKE, FAKE,
                                                  o.get("ks"), o.get("vs"), 1.0, 1.0, 100, FAKE, 8, 0.0625, 1,
                                                  FAKE, None, None, None, None, None)
    assert g16(E.QKV_BF16) == E.QKV_ERR_ARG  # a bf16 pool needs a bf16 query
    assert g16(E.QKV_F16, rows=0) == E.QKV_OK
    assert g16(E.QKV_INT8_SIDE, rows=0, ks=FAKE, vs=FAKE) == E.QKV_OK
    assert g16(E.QKV_INT8_SIDE) == E.QKV_ERR_ARG  # side scales still required
    assert _gather(lib, fmt=E.QKV_F16, ks=None, vs=None, rows=0) == E.QKV_ERR_ARG  # fp16 pool, bf16 query
    w8 = L.qkv_write_int8_f16(FAKE, FAKE, 3, 1, 64, 256, FAKE, E.QKV_INT8_SIDE, FAKE, FAKE, FAKE, FAKE, 10, None, None)
    assert w8 == E.QKV_ERR_UNSUPPORTED
    we = L.qkv_write_e4m3_f16(FAKE, FAKE, 3, 1, 256, 256, FAKE, FAKE, FAKE, 0.0, 1.0, 10, None, None)
    assert we == E.QKV_ERR_SCALE
    assert L.qkv_calib_stats_f16(FAKE, -2.0, FAKE, None) == E.QKV_ERR_SCALE


def test_varlen_host_validation(lib):
    E, L = lib, lib.lib
    vl = lambda **o: L.qsa_gather_attn_varlen(FAKE, o.get("rows", 4), 16, 1, 256, E.QKV_INT8_SIDE, FAKE, FAKE, FAKE,
                                              FAKE, 1.0, 1.0, 100, FAKE, 8, o.get("lens", FAKE), 0.0625, 1, FAKE,
                                              None, None, None, None, None)
    assert vl(lens=None) == E.QKV_ERR_ARG
    assert vl(lens=FAKE + 2) == E.QKV_ERR_ALIGN
    assert vl(rows=0) == E.QKV_OK


def test_gather_desc_layout_matches_the_header(lib, tmp_path):
    """The binding's ctypes mirror of qsa_gather_desc has the C compiler's field offsets."""
    import ctypes
    import shutil
    import subprocess
    cc = shutil.which("cc") or shutil.which("gcc")
    if cc is None:
        pytest.skip("no C compiler")
    names = [f[0] for f in lib.GatherDesc._fields_]
    src = tmp_path / "layout.c"
    src.write_text('#include <stdio.h>\n#include <stddef.h>\n#include "qkv.h"\nint main(void) {\n'
                   + "".join(f'  printf("%zu\\n", offsetof(qsa_gather_desc, {n}));\n' for n in names)
                   + '  printf("%zu\\n", sizeof(qsa_gather_desc));\n  return 0;\n}\n')
    exe = tmp_path / "layout"
    subprocess.run([cc, "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True)
    got = [int(x) for x in subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split()]
    want = [getattr(lib.GatherDesc, n).offset for n in names] + [ctypes.sizeof(lib.GatherDesc)]
    assert got == want


def test_gather_ex_host_validation(lib):
    import ctypes
    E, L = lib, lib.lib
    d = lib.GatherDesc()
    d.size = ctypes.sizeof(d)
    d.q, d.rows, d.num_q_heads, d.num_kv_heads, d.head_dim, d.fmt = FAKE, 4, 16, 1, 256, E.QKV_INT8_SIDE
    d.k_cache = d.v_cache = d.k_scale_tok = d.v_scale_tok = d.topk_idx = d.out = FAKE
    d.num_slots, d.topk, d.softmax_scale, d.num_splits = 100, 8, 0.0625, 1
    d.rows = 0
    assert L.qsa_gather_attn_ex(ctypes.byref(d), None) == E.QKV_OK
    d.size = 8
    assert L.qsa_gather_attn_ex(ctypes.byref(d), None) == E.QKV_ERR_ARG  # layout check
    d.size = ctypes.sizeof(d)
    d.q_fp16 = 2
    assert L.qsa_gather_attn_ex(ctypes.byref(d), None) == E.QKV_ERR_ARG
    d.q_fp16, d.rows, d.row_seq = 0, 4, FAKE  # row_seq without a block table
    assert L.qsa_gather_attn_ex(ctypes.byref(d), None) == E.QKV_ERR_ARG
    d.row_seq, d.block_table, d.num_seqs, d.max_blocks, d.block_size, d.q_fp16 = FAKE, FAKE, 2, 8, 16, 1
    assert L.qsa_gather_attn_ex(ctypes.byref(d), None) == E.QKV_ERR_ARG  # paged pools take a bf16 query
    assert L.qsa_gather_attn_ex(None, None) == E.QKV_ERR_ARG


def test_gather_ex_engine_selection_host_validation(lib):
    """The tensor-memory engine serves only the int8 side pool, head_dim 256, G <= 16, a bf16
    query, unpaged and unfused; everything else is refused before any launch."""
    import ctypes
    E, L = lib, lib.lib

    def desc(**kw):
        d = lib.GatherDesc()
        d.size = ctypes.sizeof(d)
        d.q, d.rows, d.num_q_heads, d.num_kv_heads, d.head_dim, d.fmt = FAKE, 4, 16, 1, 256, E.QKV_INT8_SIDE
        d.k_cache = d.v_cache = d.k_scale_tok = d.v_scale_tok = d.topk_idx = d.out = FAKE
        d.num_slots, d.topk, d.softmax_scale, d.num_splits = 100, 8, 0.0625, 1
        d.k_scale_layer = d.v_scale_layer = 1.0
        d.engine = E.QSA_ENGINE_TCGEN05
        for k, v in kw.items():
            setattr(d, k, v)
        return L.qsa_gather_attn_ex(ctypes.byref(d), None)

    assert desc(engine=2) == E.QKV_ERR_ARG
    assert desc(engine=-1) == E.QKV_ERR_ARG
    assert desc(fmt=E.QKV_E4M3, k_scale_tok=None, v_scale_tok=None) == E.QKV_ERR_UNSUPPORTED
    assert desc(fmt=E.QKV_BF16, k_scale_tok=None, v_scale_tok=None) == E.QKV_ERR_UNSUPPORTED
    assert desc(head_dim=128) == E.QKV_ERR_UNSUPPORTED
    assert desc(num_q_heads=32) == E.QKV_ERR_UNSUPPORTED  # G = 32
    assert desc(q_fp16=1) == E.QKV_ERR_UNSUPPORTED
    assert desc(block_table=FAKE, row_seq=FAKE, num_seqs=2, max_blocks=8, block_size=16) == E.QKV_ERR_UNSUPPORTED
    assert desc(num_splits=2, o_part=FAKE, lse_part=FAKE, counters=FAKE) == E.QKV_ERR_UNSUPPORTED
    assert desc(rows=0) == E.QKV_OK  # nothing to do: no launch
    # the persistent grid needs its scheduling counter: present and 4-byte aligned
    P = E.QSA_ENGINE_PERSISTENT
    assert desc(engine=P, sched=None) == E.QKV_ERR_ARG
    assert desc(engine=P, sched=FAKE + 2) == E.QKV_ERR_ALIGN
    assert desc(engine=P, sched=None, rows=0) == E.QKV_OK
    # a slot-range shard: the flag, its first slot, and the combinations it does not take
    D0 = E.QSA_ENGINE_DEFAULT
    assert desc(engine=D0, shard=2) == E.QKV_ERR_ARG
    assert desc(engine=D0, shard=1, slot_lo=-1) == E.QKV_ERR_ARG
    assert desc(engine=D0, shard=1, slot_lo=2 ** 31) == E.QKV_ERR_ARG
    assert desc(engine=D0, shard=1, slot_lo=0, block_table=FAKE, row_seq=FAKE, num_seqs=2, max_blocks=8,
                block_size=16) == E.QKV_ERR_ARG
    assert desc(engine=E.QSA_ENGINE_TCGEN05, shard=1, slot_lo=100) == E.QKV_ERR_UNSUPPORTED


def test_write_desc_layout_matches_the_header(lib, tmp_path):
    """The binding's ctypes mirror of qkv_write_desc has the C compiler's field offsets."""
    import ctypes
    import shutil
    import subprocess
    cc = shutil.which("cc") or shutil.which("gcc")
    if cc is None:
        pytest.skip("no C compiler")
    names = [f[0] for f in lib.WriteDesc._fields_]
    src = tmp_path / "wlayout.c"
    src.write_text('#include <stdio.h>\n#include <stddef.h>\n#include "qkv.h"\nint main(void) {\n'
                   + "".join(f'  printf("%zu\\n", offsetof(qkv_write_desc, {n}));\n' for n in names)
                   + '  printf("%zu\\n", sizeof(qkv_write_desc));\n  return 0;\n}\n')
    exe = tmp_path / "wlayout"
    subprocess.run([cc, "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True)
    got = [int(x) for x in subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split()]
    want = [getattr(lib.WriteDesc, n).offset for n in names] + [ctypes.sizeof(lib.WriteDesc)]
    assert got == want


def test_write_ex_host_validation(lib):
    """Refusals before any launch: descriptor size, one addressing at a time, paged geometry,
    format-specific scales."""
    import ctypes
    E = lib

    def call(**over):
        d = lib.WriteDesc()
        d.size = ctypes.sizeof(lib.WriteDesc)
        d.fmt, d.act_fp16 = E.QKV_INT8_SIDE, 0
        d.k = d.v = FAKE
        d.num_tokens, d.num_kv_heads, d.head_dim, d.token_stride = 3, 1, 256, 256
        d.slot_mapping = FAKE
        d.k_cache = d.v_cache = FAKE
        d.k_scale = d.v_scale = FAKE
        d.k_scale_layer = d.v_scale_layer = 1.0
        d.num_slots = 10
        for k, v in over.items():
            setattr(d, k, v)
        return lib.lib.qkv_write_ex(ctypes.byref(d), None)

    assert lib.lib.qkv_write_ex(None, None) == E.QKV_ERR_ARG
    assert call(size=8) == E.QKV_ERR_ARG
    assert call(fmt=E.QKV_BF16) == E.QKV_ERR_ARG
    assert call(act_fp16=2) == E.QKV_ERR_ARG
    assert call(token_seq=FAKE) == E.QKV_ERR_ARG  # slot ids and a paged pool at once
    paged = dict(slot_mapping=None, token_seq=FAKE, token_pos=FAKE, block_table=FAKE, num_seqs=2, max_blocks=4,
                 block_size=16)
    assert call(**{**paged, "block_table": None}) == E.QKV_ERR_ARG
    assert call(**{**paged, "block_size": 0}) == E.QKV_ERR_ARG
    assert call(**{**paged, "max_blocks": 1 << 20, "block_size": 1 << 12}) == E.QKV_ERR_ARG  # positions past 2^31
    assert call(**{**paged, "token_pos": FAKE + 2}) == E.QKV_ERR_ALIGN
    assert call(fmt=E.QKV_E4M3) == E.QKV_ERR_ARG  # E4M3 takes no per-token scale tensors
    assert call(fmt=E.QKV_E4M3, k_scale=None, v_scale=None, k_scale_layer=0.0) == E.QKV_ERR_SCALE
    assert call(fmt=E.QKV_INT8_INLINE) == E.QKV_ERR_ARG  # inline records hold their scales
    assert call(num_tokens=0) == E.QKV_OK
    assert call(**{**paged, "num_tokens": 0}) == E.QKV_OK


def test_noalloc_rejects_sizes_beyond_its_scratch_before_any_cuda_call(lib):
    """The no-allocation split gather bounds each factor of its partials' size before it
    multiplies them, so no product can wrap past the check (num_q_heads alone may be large)."""
    L = lib.lib

    def call(rows, hq, P, hkv=1):
        return L.qsa_gather_attn_splitk_noalloc(FAKE, rows, hq, hkv, 256, lib.QKV_INT8_SIDE, FAKE, FAKE, FAKE, FAKE,
                                                1.0, 1.0, 100, FAKE, 8, 0.0625, P, FAKE, None, None, None)

    big = 2 ** 31 - 1
    assert call(2 ** 20, big, 2 ** 20) == lib.QKV_ERR_ARG  # the 64-bit product would wrap
    assert call(2 ** 24, 16, 2 ** 24) == lib.QKV_ERR_ARG
    assert call(1, big, 2) == lib.QKV_ERR_ARG
    assert call(2 ** 25, 16, 2) == lib.QKV_ERR_ARG
    assert call(64, 16, 16) == lib.QKV_ERR_ARG  # 64 x 16 x 16 x 257 x 4 B: just past 16 MiB
    assert call(0, 16, 8) == lib.QKV_OK  # nothing to do, nothing launched
