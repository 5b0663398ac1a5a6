"""Seeded synthetic workloads for the quantized KV-cache write and the top-k gather decode.

This module only draws inputs. It holds none of the method's arithmetic (no quantisation,
no scale rule, no attention): it returns bf16 bit patterns for K, V and q, slot mappings
and top-k index lists, drawn from numpy's PCG64 generator in a fixed order. The CPU oracle
and the CUDA path both consume exactly what it returns.

Draw order inside one workload (one ``np.random.default_rng(seed)`` stream):
pool K, pool V, outlier choice, slot permutation, q, top-k lists, then any extra
per-step tensors. Normals are float32 standard normals, scaled (outliers) in float32 and
rounded to bf16 with round-to-nearest-even. Config 3's layers each use their own stream,
``default_rng([seed, layer])``.

Workload shapes follow the page workloads:
* int8 per-(token,head) KV cache for the Qwen3.8-Flash-Next QSA path, §The finding worth
  upstreaming: 2048 query rows gathering top-k 1024 scattered slots; one KV head of
  head_dim 256 (256 B of int8 data per head).
* [Model][SM70][FP8] Add calibrated E4M3 QSA KV cache / [Perf][SM70][FP8] Hoist QSA E4M3 KV
  scales, §Test plan / §Changes: 24 per-layer scalars (12 layers x K,V); a long top-k 2051
  split-K shape.
* SuperPUPS/Qwen3.8-Flash-Next-INT8KV, §What it buys you: MTP k=4 decode (5 query
  positions per sequence).
* [Model][SM70][FP8] Add calibrated E4M3 QSA KV cache, §Implementation scope and §Targeted
  mixed-batch scheduler regression: a 49-row batch of a 46-row catch-up chunk plus three
  decode rows; batches split into a bulk and tails of at most 16 rows.
"""

from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np

HEAD_DIM = 256


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (nearest, ties to even) and return the uint16 bits.

    Inputs are finite by construction here, so no NaN handling is needed.
    """
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).reshape(-1)
    out = np.empty(u.shape, dtype=np.uint16)
    step = 1 << 20  # chunked so the temporaries stay in cache
    for a in range(0, u.size, step):
        c = u[a:a + step]
        lsb = (c >> np.uint32(16)) & np.uint32(1)
        out[a:a + step] = (c + np.uint32(0x7FFF) + lsb) >> np.uint32(16)
    return out.reshape(np.shape(x))


def f32_to_f16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to IEEE half (numpy's conversion: nearest, ties to even) and
    return the uint16 bits. Inputs here are finite and far below the fp16 range's end."""
    return np.ascontiguousarray(x, dtype=np.float32).astype(np.float16).view(np.uint16)


@dataclasses.dataclass
class Workload:
    """One synthetic problem: tokens written into a slot pool, then query rows gathering it."""

    name: str
    seed: int
    num_slots: int
    num_kv_heads: int
    num_q_heads: int
    head_dim: int
    k_tokens: np.ndarray  # uint16 bf16 bits [T, Hkv, D]
    v_tokens: np.ndarray  # uint16 bf16 bits [T, Hkv, D]
    slot_mapping: np.ndarray  # int64 [T], token -> slot, -1 = skip
    q: np.ndarray  # uint16 bf16 bits [R, Hq, D]
    topk: Optional[np.ndarray]  # int32 [R, k], slot ids, -1 = padding (None: paged rows only)
    softmax_scale: float
    num_splits: int = 1
    # Per-step write of new tokens (decode step): bf16 bits [Tn, Hkv, D] and slots [Tn].
    step_k: Optional[np.ndarray] = None
    step_v: Optional[np.ndarray] = None
    step_slots: Optional[np.ndarray] = None
    # Paged pools: block table int32 [num_seqs, max_blocks], each row's sequence int32 [R] and
    # its entries as logical positions int32 [R, k] (-1 = padding), blocks of block_size slots.
    block_table: Optional[np.ndarray] = None
    row_seq: Optional[np.ndarray] = None
    topk_pos: Optional[np.ndarray] = None
    block_size: int = 0
    notes: str = ""
    # 16-bit type of q and of the new K/V tokens: "bf16", or "f16" for the FP16-activation
    # contract of "[Model][SM70][FP8] Add calibrated E4M3 QSA KV cache" (§Purpose)
    act_dtype: str = "bf16"
    # Rows of different lengths (the varlen launch): valid entries per row int32 [R]; entries
    # of row r past row_len[r] are -1.
    row_len: Optional[np.ndarray] = None

    @property
    def rows(self) -> int:
        return int((self.topk if self.topk is not None else self.topk_pos).shape[0])

    @property
    def topk_len(self) -> int:
        return int(self.topk.shape[1])


def _normals(rng: np.random.Generator, shape, chunk_rows: int = 65536) -> np.ndarray:
    """float32 standard normals drawn in row chunks (same stream as one big draw)."""
    out = np.empty(shape, dtype=np.float32)
    flat = out.reshape(shape[0], -1)
    for a in range(0, shape[0], chunk_rows):
        b = min(shape[0], a + chunk_rows)
        flat[a:b] = rng.standard_normal((b - a, flat.shape[1]), dtype=np.float32)
    return out


def _distinct_rows(rng: np.random.Generator, rows: int, population: int, k: int) -> np.ndarray:
    """`rows` lists of `k` distinct integers uniform over [0, population), in random order.

    Each row keeps the first k distinct values of an i.i.d. uniform integer stream, which is
    a uniformly random k-subset in uniformly random order. Streams are drawn 2k at a time
    per row; a row that is still short draws again. For k > population / 4 a permutation is
    used instead.
    """
    out = np.empty((rows, k), dtype=np.int64)
    if k * 4 > population:
        for r in range(rows):
            out[r] = rng.permutation(population)[:k]
        return out
    draws = rng.integers(0, population, size=(rows, 2 * k), dtype=np.int64)
    for r in range(rows):
        seq = draws[r]
        while True:
            _, first = np.unique(seq, return_index=True)
            if first.size >= k:
                out[r] = seq[np.sort(first)[:k]]
                break
            seq = np.concatenate([seq, rng.integers(0, population, size=2 * k, dtype=np.int64)])
    return out


def _scaled_bf16(base: np.ndarray, factor: np.ndarray) -> np.ndarray:
    """Multiply token vectors by per-token factors in float32, then round to bf16 bits."""
    return f32_to_bf16_bits(base * factor.reshape((-1,) + (1,) * (base.ndim - 1)))


def tiny(seed: int = 0) -> Workload:
    """Tiny int8 sparse decode: 4096 slots, GQA 8, 16 rows x top-k 64, every 64th token x20."""
    S, H, D, G, R, K = 4096, 1, HEAD_DIM, 8, 16, 64
    rng = np.random.default_rng(seed)
    k = _normals(rng, (S, H, D))
    v = _normals(rng, (S, H, D))
    factor = np.ones(S, dtype=np.float32)
    factor[np.arange(S) % 64 == 0] = np.float32(20.0)
    slot_mapping = rng.permutation(S).astype(np.int64)
    q = f32_to_bf16_bits(_normals(rng, (R, H * G, D)))
    topk = _distinct_rows(rng, R, S, K).astype(np.int32)
    return Workload("tiny int8 sparse decode (S=4096, G=8, R=16, k=64)", seed, S, H, H * G, D,
                    _scaled_bf16(k, factor), _scaled_bf16(v, factor), slot_mapping, q, topk,
                    softmax_scale=1.0 / 16.0, num_splits=1)


def page1_shape(seed: int = 1, rows: int = 2048, topk: int = 1024, num_slots: int = 262144,
                with_step: bool = True) -> Workload:
    """2048 rows x top-k 1024 over a 262144-slot pool, G=16, 1% outlier tokens x16.

    With `with_step`, also draws one decode step's worth of new tokens (one per row) and
    distinct destination slots for them.
    """
    S, H, D, G = num_slots, 1, HEAD_DIM, 16
    rng = np.random.default_rng(seed)
    k = _normals(rng, (S, H, D))
    v = _normals(rng, (S, H, D))
    n_out = int(round(0.01 * S))
    outliers = rng.choice(S, size=n_out, replace=False)
    factor = np.ones(S, dtype=np.float32)
    factor[outliers] = np.float32(16.0)
    slot_mapping = rng.permutation(S).astype(np.int64)
    q = f32_to_bf16_bits(_normals(rng, (rows, H * G, D)))
    idx = _distinct_rows(rng, rows, S, topk).astype(np.int32)
    wl = Workload(f"page-1 shape (S={S}, G=16, R={rows}, k={topk})", seed, S, H, H * G, D,
                  _scaled_bf16(k, factor), _scaled_bf16(v, factor), slot_mapping, q, idx,
                  softmax_scale=1.0 / 16.0, num_splits=1)
    if with_step:
        wl.step_k = f32_to_bf16_bits(_normals(rng, (rows, H, D)))
        wl.step_v = f32_to_bf16_bits(_normals(rng, (rows, H, D)))
        wl.step_slots = rng.choice(S, size=rows, replace=False).astype(np.int64)
    return wl


def e4m3_splitk_layer(layer: int, seed: int = 2, rows: int = 64, topk: int = 2051,
                      num_slots: int = 131072, num_splits: int = 8) -> Workload:
    """One of 12 layers: its own 131072-slot pool and q; 64 rows x top-k 2051, 8 K-splits."""
    S, H, D, G = num_slots, 1, HEAD_DIM, 16
    rng = np.random.default_rng([seed, layer])
    k = f32_to_bf16_bits(_normals(rng, (S, H, D)))
    v = f32_to_bf16_bits(_normals(rng, (S, H, D)))
    slot_mapping = rng.permutation(S).astype(np.int64)
    q = f32_to_bf16_bits(_normals(rng, (rows, H * G, D)))
    idx = _distinct_rows(rng, rows, S, topk).astype(np.int32)
    return Workload(f"calibrated E4M3 split-K layer {layer} (S={S}, R={rows}, k={topk}, P={num_splits})",
                    seed, S, H, H * G, D, k, v, slot_mapping, q, idx,
                    softmax_scale=1.0 / 16.0, num_splits=num_splits)


E4M3_SPLITK_LAYERS = 12


def long_context_decode(seed: int = 3, num_seqs: int = 8, context: int = 131072, block: int = 16,
                        rows_per_seq: int = 5, topk: int = 2048, recent: int = 4096,
                        recent_picks: int = 1536, num_splits: int = 16) -> Workload:
    """8 sequences x 131072 tokens in a paged pool (blocks of 16, randomly permuted).

    Each sequence has 5 query rows (MTP k=4); each row draws 1536 distinct positions from
    the sequence's last 4096 tokens and 512 distinct positions from the rest. Positions
    map to physical slots through the permuted block table here, so the kernel takes slot ids.
    """
    H, D, G = 1, HEAD_DIM, 16
    n_blocks_seq = context // block
    total_blocks = num_seqs * n_blocks_seq
    S = total_blocks * block
    rng = np.random.default_rng(seed)
    k = f32_to_bf16_bits(_normals(rng, (S, H, D)))
    v = f32_to_bf16_bits(_normals(rng, (S, H, D)))
    block_perm = rng.permutation(total_blocks).astype(np.int64)
    # token (b, pos) is token index b*context + pos; its slot via the block table
    pos = np.arange(context, dtype=np.int64)
    slot_mapping = np.empty(S, dtype=np.int64)
    for b in range(num_seqs):
        phys = block_perm[b * n_blocks_seq + pos // block]
        slot_mapping[b * context:(b + 1) * context] = phys * block + pos % block
    R = num_seqs * rows_per_seq
    q = f32_to_bf16_bits(_normals(rng, (R, H * G, D)))
    idx = np.empty((R, topk), dtype=np.int32)
    pos_out = np.empty((R, topk), dtype=np.int32)
    older = context - recent
    for b in range(num_seqs):
        base = b * context
        for j in range(rows_per_seq):
            r = b * rows_per_seq + j
            near = older + rng.choice(recent, size=recent_picks, replace=False)
            far = rng.choice(older, size=topk - recent_picks, replace=False)
            positions = np.concatenate([near, far])
            idx[r] = slot_mapping[base + positions]
            pos_out[r] = positions
    block_table = block_perm.reshape(num_seqs, n_blocks_seq).astype(np.int32)
    row_seq = np.repeat(np.arange(num_seqs, dtype=np.int32), rows_per_seq)
    return Workload(f"long-context decode (8 x {context} ctx, paged blocks of {block}, R={R}, k={topk})",
                    seed, S, H, H * G, D, k, v, slot_mapping, q, idx,
                    softmax_scale=1.0 / 16.0, num_splits=num_splits,
                    block_table=block_table, row_seq=row_seq, topk_pos=pos_out, block_size=block,
                    notes="topk holds the slot ids placed by the generator; topk_pos/block_table/row_seq "
                          "give the same rows as logical positions of a paged pool")


def chunked_prefill(seed: int = 4, new_tokens: int = 8192, num_slots: int = 524288,
                    topk: int = 1024) -> Workload:
    """8192 new tokens scattered into a 524288-slot pool; row i attends min(1024, i) positions < i.

    Row 0 has no valid index (all -1). Padding entries are -1.
    """
    H, D, G = 1, HEAD_DIM, 16
    T, S = new_tokens, num_slots
    rng = np.random.default_rng(seed)
    k = f32_to_bf16_bits(_normals(rng, (T, H, D)))
    v = f32_to_bf16_bits(_normals(rng, (T, H, D)))
    slot_mapping = rng.choice(S, size=T, replace=False).astype(np.int64)
    q = f32_to_bf16_bits(_normals(rng, (T, H * G, D)))
    idx = np.full((T, topk), -1, dtype=np.int32)
    for i in range(1, T):
        n = min(topk, i)
        positions = rng.choice(i, size=n, replace=False)
        idx[i, :n] = slot_mapping[positions]
    return Workload(f"chunked-prefill write + causal sparse attention (T={T}, S={S}, k={topk})",
                    seed, S, H, H * G, D, k, v, slot_mapping, q, idx,
                    softmax_scale=1.0 / 16.0, num_splits=1)


def small_random(seed: int, num_slots: int, rows: int, topk: int, num_q_heads: int = 16,
                 num_kv_heads: int = 1, pad_frac: float = 0.0, outlier_frac: float = 0.0,
                 outlier_factor: float = 16.0, num_tokens: Optional[int] = None,
                 num_splits: int = 1, softmax_scale: float = 1.0 / 16.0,
                 zero_tokens: int = 0, act_dtype: str = "bf16", head_dim: int = HEAD_DIM) -> Workload:
    """Generic small case for parity tests: ragged top-k, -1 padding, optional outliers.

    `zero_tokens` tokens (chosen after the outliers) get all-zero K and V vectors, the
    degenerate absmax = 0 case. act_dtype 'f16' rounds q, K and V to IEEE half instead of
    bf16 (same draws). head_dim 128 draws 128-wide heads instead of 256.
    """
    S, H, D = num_slots, num_kv_heads, head_dim
    T = S if num_tokens is None else num_tokens
    rng = np.random.default_rng(seed)
    k = _normals(rng, (T, H, D))
    v = _normals(rng, (T, H, D))
    factor = np.ones(T, dtype=np.float32)
    n_out = int(round(outlier_frac * T))
    if n_out:
        factor[rng.choice(T, size=n_out, replace=False)] = np.float32(outlier_factor)
    if zero_tokens:
        factor[rng.choice(T, size=zero_tokens, replace=False)] = np.float32(0.0)
    slot_mapping = rng.choice(S, size=T, replace=False).astype(np.int64)
    to16 = f32_to_f16_bits if act_dtype == "f16" else f32_to_bf16_bits
    q = to16(_normals(rng, (rows, num_q_heads, D)))
    written = slot_mapping
    kk = min(topk, T)
    idx = np.full((rows, topk), -1, dtype=np.int32)
    for r in range(rows):
        picks = written[rng.choice(T, size=kk, replace=False)]
        if pad_frac > 0:
            drop = rng.random(kk) < pad_frac
            picks = np.where(drop, -1, picks)
        idx[r, :kk] = picks
    if act_dtype == "f16":
        kt, vt = to16(k * factor[:, None, None]), to16(v * factor[:, None, None])
    else:
        kt, vt = _scaled_bf16(k, factor), _scaled_bf16(v, factor)
    return Workload(f"small random (S={S}, T={T}, R={rows}, k={topk}, Hq={num_q_heads}, Hkv={H}, {act_dtype})",
                    seed, S, H, num_q_heads, D, kt, vt,
                    slot_mapping, q, idx, softmax_scale=softmax_scale, num_splits=num_splits, act_dtype=act_dtype)



def small_paged(seed: int, num_seqs: int = 3, max_blocks: int = 6, block_size: int = 16, rows: int = 5,
                topk: int = 40, pad_frac: float = 0.1, unallocated_frac: float = 0.15,
                num_q_heads: int = 16, num_kv_heads: int = 1, head_dim: int = HEAD_DIM) -> Workload:
    """A small paged pool: num_seqs x max_blocks blocks of block_size slots, each sequence's
    blocks a random permutation of the pool's blocks, some table entries unallocated (-1).

    Rows draw distinct positions of their sequence (some landing in unallocated blocks, which
    the library must flag) plus -1 padding. Slot ids are left to the oracle's translation.
    """
    H, D, Hq = num_kv_heads, head_dim, num_q_heads
    rng = np.random.default_rng(seed)
    total_blocks = num_seqs * max_blocks
    S = total_blocks * block_size
    k = f32_to_bf16_bits(_normals(rng, (S, H, D)))
    v = f32_to_bf16_bits(_normals(rng, (S, H, D)))
    slot_mapping = np.arange(S, dtype=np.int64)  # token t lives in slot t
    table = rng.permutation(total_blocks).astype(np.int32).reshape(num_seqs, max_blocks)
    table[rng.random(table.shape) < unallocated_frac] = -1
    q = f32_to_bf16_bits(_normals(rng, (rows, Hq, D)))
    row_seq = rng.integers(0, num_seqs, size=rows).astype(np.int32)
    pos = np.empty((rows, topk), dtype=np.int32)
    for r in range(rows):
        pos[r] = rng.choice(max_blocks * block_size, size=topk, replace=False)
        pos[r, rng.random(topk) < pad_frac] = -1
    return Workload(f"small paged pool (seed {seed}, {num_seqs} seqs x {max_blocks} blocks of {block_size})",
                    seed, S, H, Hq, D, k, v, slot_mapping, q, None, softmax_scale=1.0 / 16.0,
                    block_table=table, row_seq=row_seq, topk_pos=pos, block_size=block_size,
                    notes="paged rows only: slot ids come from the block table")

def cancelling_pairs(seed: int = 8, rows: int = 32, background: int = 300, num_slots: int = 8192,
                     pair_gain: float = 4.0, v_gain: float = 16.0) -> Workload:
    """Rows whose output is a near cancellation of two outlier keys.

    Row r gathers its own pair of tokens A_r, B_r plus `background` distinct ordinary tokens,
    in random order. A_r's K is pair_gain x a normal vector and B_r's K equals it, except that
    one coordinate is scaled by (1 + eps), eps cycling through 0, 2^-7, 2^-5 and 2^-3 (an
    exact tie, then ever larger gaps). Their V vectors are v_gain x a normal vector and its
    exact negation. Every head's q is A_r's K times 16 L / |K|^2 plus N(0, 0.2) noise, so the
    pair's logits sit ~L above the rest (softmax scale 1/16), L = 8 (the other keys still
    count) or 40 (only the pair does; outlier keys reach such logits on the pages' data,
    gain 16 x a normal vector against a normal q). The output is the small difference of two
    large, nearly equal terms: only logits accurate to ~1e-6 keep it within 5e-5, and at
    L = 40 the rounding of an fp32 logit alone exceeds that.
    """
    S, H, G, D = num_slots, 1, 16, HEAD_DIM
    T = S
    rng = np.random.default_rng(seed)
    k = _normals(rng, (T, H, D))
    v = _normals(rng, (T, H, D))
    eps = np.array([0.0, 2.0 ** -7, 2.0 ** -5, 2.0 ** -3], dtype=np.float32)
    q = np.empty((rows, H * G, D), dtype=np.float32)
    for r in range(rows):
        a, b = 2 * r, 2 * r + 1
        k[a] *= np.float32(pair_gain)
        k[b] = k[a]
        d = int(rng.integers(D))
        k[b, 0, d] = k[a, 0, d] * (np.float32(1.0) + eps[r % eps.size])
        v[a] *= np.float32(v_gain)
        v[b] = -v[a]
        ka = k[a, 0]
        gap = 8.0 if (r // eps.size) % 2 == 0 else 40.0
        q[r] = ka[None, :] * np.float32(16.0 * gap / float(ka @ ka)) + np.float32(0.2) * rng.standard_normal(
            (H * G, D), dtype=np.float32)
    slot_mapping = rng.permutation(S).astype(np.int64)
    idx = np.empty((rows, background + 2), dtype=np.int32)
    for r in range(rows):
        others = 2 * rows + rng.choice(T - 2 * rows, size=background, replace=False)
        toks = rng.permutation(np.concatenate([[2 * r, 2 * r + 1], others]))
        idx[r] = slot_mapping[toks]
    return Workload(f"cancelling outlier pairs (S={S}, R={rows}, k={background + 2})", seed, S, H, H * G, D,
                    f32_to_bf16_bits(k), f32_to_bf16_bits(v), slot_mapping, f32_to_bf16_bits(q), idx,
                    softmax_scale=1.0 / 16.0,
                    notes="pair tokens 2r, 2r + 1 per row r; K_B = K_A up to one coordinate, V_B = -V_A")


def mixed_catchup_decode(seed: int = 6, catchup_rows: int = 46, catchup_start: int = 64,
                         decode_rows: int = 3, decode_context: int = 8192, topk: int = 2051,
                         num_slots: int = 131072) -> Workload:
    """A 49-row mixed batch: a 46-row catch-up chunk of one request plus three decode rows.

    The catch-up chunk covers positions catchup_start .. catchup_start + 45 of its request, and
    its row i attends every earlier position (catchup_start + i keys: short rows). Each decode
    row belongs to a request of decode_context tokens and attends top-k 2051 distinct positions
    of it. Every token of the four requests is written to its own slot of a shared pool; the
    rows list slot ids, with -1 past each row's length (row_len).
    """
    H, D, G = 1, HEAD_DIM, 16
    n_cu = catchup_start + catchup_rows
    T = n_cu + decode_rows * decode_context
    rng = np.random.default_rng(seed)
    k = f32_to_bf16_bits(_normals(rng, (T, H, D)))
    v = f32_to_bf16_bits(_normals(rng, (T, H, D)))
    slot_mapping = rng.choice(num_slots, size=T, replace=False).astype(np.int64)
    R = catchup_rows + decode_rows
    q = f32_to_bf16_bits(_normals(rng, (R, H * G, D)))
    idx = np.full((R, topk), -1, dtype=np.int32)
    lens = np.zeros(R, dtype=np.int32)
    for i in range(catchup_rows):
        n = min(topk, catchup_start + i)
        idx[i, :n] = slot_mapping[rng.permutation(catchup_start + i)[:n]]
        lens[i] = n
    for j in range(decode_rows):
        base = n_cu + j * decode_context
        idx[catchup_rows + j] = slot_mapping[base + rng.choice(decode_context, size=topk, replace=False)]
        lens[catchup_rows + j] = topk
    return Workload(f"mixed catch-up/decode batch ({catchup_rows} catch-up rows of "
                    f"{catchup_start}..{n_cu - 1} keys + {decode_rows} decode rows of top-k {topk})",
                    seed, num_slots, H, H * G, D, k, v, slot_mapping, q, idx,
                    softmax_scale=1.0 / 16.0, num_splits=8, row_len=lens)


def bulk_tail_decode(seed: int = 7, bulk_rows: int = 48, tail_rows: int = 13, topk: int = 2051,
                     num_slots: int = 131072) -> Workload:
    """A 16-divisible bulk of 48 full rows (top-k 2051) followed by a 13-row tail of mixed lengths.

    Tail row j attends a length drawn uniformly from 1 .. 2051 (one tail row is forced to 1,
    one to the full 2051). All rows gather distinct slots of one 131072-slot pool.
    """
    H, D, G = 1, HEAD_DIM, 16
    rng = np.random.default_rng(seed)
    k = f32_to_bf16_bits(_normals(rng, (num_slots, H, D)))
    v = f32_to_bf16_bits(_normals(rng, (num_slots, H, D)))
    slot_mapping = rng.permutation(num_slots).astype(np.int64)
    R = bulk_rows + tail_rows
    q = f32_to_bf16_bits(_normals(rng, (R, H * G, D)))
    idx = _distinct_rows(rng, R, num_slots, topk).astype(np.int32)
    lens = np.full(R, topk, dtype=np.int32)
    lens[bulk_rows:] = rng.integers(1, topk + 1, tail_rows)
    lens[bulk_rows] = 1
    lens[bulk_rows + 1] = topk
    for r in range(bulk_rows, R):
        idx[r, lens[r]:] = -1
    return Workload(f"bulk + tail decode batch ({bulk_rows} rows of top-k {topk} + {tail_rows} tail rows "
                    f"of mixed length)", seed, num_slots, H, H * G, D, k, v, slot_mapping, q, idx,
                    softmax_scale=1.0 / 16.0, num_splits=8, row_len=lens)


CONFIGS = {
    1: tiny,
    2: page1_shape,
    3: e4m3_splitk_layer,
    4: long_context_decode,
    5: chunked_prefill,
}
