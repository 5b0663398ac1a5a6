"""CPU oracle for the quantized KV-cache write and the top-k gather decode.

TEST INFRASTRUCTURE ONLY. Only the tests, the package smoke check and the benchmark's CPU
baseline leg may import this package; the product path never does, and it shares no code,
constants or helpers with the CUDA library.

It is written to be read against the pages, not to be fast:

* quant.py     int8 per-(token,head) absmax/127 quantisation, the FP8 E4M3 encoder/decoder
               and the calibrated per-layer scale amax/448, plus the slot-pool writes in the
               three stored layouts (int8 with side scales, int8 with inline 260 B records,
               E4M3 bytes).
* attention.py fp64 dequantisation of a slot pool, top-k gather attention with a
               max-subtracted softmax, the split-K partition and the log-sum-exp merge.
* paging.py    logical positions of a paged pool -> slot ids through a block table.
* calibration.py  per-tensor calibration statistics: max-abs, nearest-rank p99.9 / p99.99 of
               |x|, the calibrated scale amax/448, and the counts of scaled magnitudes below
               E4M3's smallest subnormal, in its subnormal range, and clipped by saturation.

Pages cited (by title):
  [INT8-PR]  "int8 per-(token,head) KV cache for the Qwen3.8-Flash-Next QSA path"
  [INT8-KV]  "SuperPUPS/Qwen3.8-Flash-Next-INT8KV" (INT8 KV build, int8_per_token_head)
  [E4M3-PR]  "[Model][SM70][FP8] Add calibrated E4M3 QSA KV cache"
  [HOIST-PR] "[Perf][SM70][FP8] Hoist QSA E4M3 KV scales"
  [SCALES]   "Qwen3.8 Flash Next NVFP4 QSA FP8 E4M3 KV Scales" (model card)

Every function is pinned by a test under tests/ that does not re-derive it (closed forms,
library routines on special cases, brute force, invariants, hand-worked fixtures).
"""

from . import attention, calibration, paging, quant  # noqa: F401
