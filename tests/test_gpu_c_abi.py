"""A decode step through the C ABI from a plain C program (GPU).

tests/c/decode_step.c includes only qkv.h and the CUDA runtime, links libqkv.so, and runs
qkv_write_int8 then qsa_gather_attn (unsplit, and split + qsa_splitk_merge) on buffers it
allocates itself. No Python and no PyTorch take part in its process. Its outputs must match
the fp64 oracle within |gpu - ref| <= 5e-5 + 1e-3 |ref|, with both status words zero.
("int8 per-(token,head) KV cache for the Qwen3.8-Flash-Next QSA path" §The finding worth
upstreaming: the write and the gather of the int8 side-tensor layout.)
"""

import os
import shutil
import subprocess

import numpy as np
import pytest

from gen import small_random
from harness import OraclePool, assert_close

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _cuda_home():
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    return os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))


def test_decode_step_from_c(tmp_path):
    import quantized_kv_cache_write_gb300 as q  # builds libqkv.so if needed
    cc = shutil.which("cc") or shutil.which("gcc")
    if cc is None:
        pytest.skip("no C compiler")
    lib_dir = os.path.dirname(q.LIB_PATH)
    cuda = _cuda_home()
    exe = tmp_path / "decode_step"
    subprocess.run([cc, "-O2", "-I", os.path.join(ROOT, "include"), "-I", os.path.join(cuda, "include"),
                    os.path.join(ROOT, "tests", "c", "decode_step.c"), "-L", lib_dir, "-lqkv",
                    "-L", os.path.join(cuda, "lib64"), "-lcudart", f"-Wl,-rpath,{lib_dir}",
                    f"-Wl,-rpath,{os.path.join(cuda, 'lib64')}", "-o", str(exe)], check=True)
    wl = small_random(61, num_slots=5000, num_tokens=4000, rows=6, topk=300, pad_frac=0.05, outlier_frac=0.02)
    T, S, R, K, Hq, D = wl.k_tokens.shape[0], wl.num_slots, wl.rows, wl.topk_len, wl.num_q_heads, wl.head_dim
    (tmp_path / "meta.txt").write_text(f"{T} {S} {R} {K} {Hq} {D}\n")
    for name, arr, dt in (("k.bin", wl.k_tokens, np.uint16), ("v.bin", wl.v_tokens, np.uint16),
                          ("slots.bin", wl.slot_mapping, np.int64), ("q.bin", wl.q, np.uint16),
                          ("idx.bin", wl.topk, np.int32)):
        np.ascontiguousarray(arr, dtype=dt).tofile(tmp_path / name)
    run = subprocess.run([str(exe), str(tmp_path)], capture_output=True, text=True, timeout=300)
    assert run.returncode == 0, run.stderr
    assert (tmp_path / "status.txt").read_text().split() == ["0", "0"]
    out = np.fromfile(tmp_path / "out.bin", dtype=np.float32).reshape(R, Hq, D)
    out_split = np.fromfile(tmp_path / "out_split.bin", dtype=np.float32).reshape(R, Hq, D)
    lse = np.fromfile(tmp_path / "lse.bin", dtype=np.float32).reshape(R, Hq)
    ro, rl = OraclePool(wl, "int8_side").attend(wl)
    assert_close(out, ro, "C ABI out")
    assert_close(out_split, ro, "C ABI split out")
    assert_close(lse, rl, "C ABI lse")
