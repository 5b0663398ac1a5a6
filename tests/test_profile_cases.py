"""The profiling driver's command line (CPU: no case is built or launched here)."""

import subprocess
import sys
import os

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_cases_and_help_without_a_gpu():
    from quantized_kv_cache_write_gb300 import profile_cases as pc
    assert {"page1_int8_side", "page1_int8_inline", "page1_e4m3", "page1_bf16", "page1_tcgen05", "e4m3_layer",
            "long_context", "chunked_prefill", "mixed_default", "mixed_persistent"} <= set(pc.CASES)
    r = subprocess.run([sys.executable, "-m", "quantized_kv_cache_write_gb300.profile_cases", "--help"], cwd=ROOT,
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and "page1_int8_side" in r.stdout
    # an unknown case is refused by the argument parser before anything is built
    r = subprocess.run([sys.executable, "-m", "quantized_kv_cache_write_gb300.profile_cases", "no_such_case"],
                       cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode != 0 and "invalid choice" in r.stderr
