"""Seeded synthetic inputs for the spec-verify workloads.

This module is shared by the tests, the benchmark and the smoke check.  It
holds only random draws, shapes and the fp32 -> bf16 storage rounding; none of
the method's arithmetic (no gating, no recurrence, no normalisation inside the
kernel's sense).  The one transformation applied to draws is the workloads'
stated input property "q, k L2-normalised" (done in fp32 before storage
rounding), which describes the input distribution, not a step of the path.

Storage conventions (numpy, host):
  * bf16 tensors are ``np.uint16`` arrays of bf16 bit patterns;
  * fp32 tensors are ``np.float32``;
  * ``to_f64`` turns either into exact fp64 values for the oracle.

Workloads (shapes and distributions of the pages' Qwen3-Next-shaped GDN layer;
the pages measure on GSM8K / AIME served by real models, which need datasets
and trained weights, so these seeded tensors stand in for them):
  C0 tiny fp32:  B=1, H=HV=2, K=V=32, T=4, L=8
  C1 Qwen3-Next: B=1, H=16, HV=32, K=V=128, T=4, L=64, bf16 I/O
  C2 batch sweep of the C1 layer: B in {8, 32, 128, 256}, 512-slot pool
  C3 flush-heavy: C1 heads, B=16, L=16, 16384 committed tokens per slot
  C4 KDA: C1 dims with a per-key-channel gate, B in {1, 64}
"""
from __future__ import annotations

import math
import zlib
from dataclasses import dataclass, field

import numpy as np

BF16 = "bf16"
FP32 = "fp32"


# ------------------------------------------------------------ storage rounding

def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16 (nearest, ties to even) and return the uint16 bits."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    rounding = ((u >> 16) & 1) + 0x7FFF
    return ((u + rounding) >> 16).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    b = np.ascontiguousarray(b, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


def store(x: np.ndarray, io_dtype: str) -> np.ndarray:
    """fp32 draws -> storage array in the I/O dtype."""
    if io_dtype == BF16:
        return f32_to_bf16_bits(x)
    if io_dtype == FP32:
        return np.ascontiguousarray(x, dtype=np.float32)
    raise ValueError(io_dtype)


def to_f64(x: np.ndarray) -> np.ndarray:
    """Exact fp64 values of a storage array (bf16 bits or fp32)."""
    if x.dtype == np.uint16:
        return bf16_bits_to_f32(x).astype(np.float64)
    return np.asarray(x, dtype=np.float64)


def _unit_rows(x: np.ndarray) -> np.ndarray:
    """Scale the last axis to unit L2 norm in fp32 (the workloads' input property)."""
    x = x.astype(np.float32)
    n = np.sqrt(np.sum(x * x, axis=-1, keepdims=True, dtype=np.float32))
    return (x / np.maximum(n, np.float32(1e-30))).astype(np.float32)


# ------------------------------------------------------------ workload shapes

@dataclass
class Workload:
    name: str
    B: int
    H: int
    HV: int
    K: int
    V: int
    T: int
    L: int
    io_dtype: str = BF16
    per_key_gate: bool = False
    num_slots: int = 0          # 0 -> B + 1 (a guard slot beyond the used ones)
    prefix: int = 0             # tokens of prefix that build the checkpoint
    rounds: int = 0
    extra: dict = field(default_factory=dict)

    @property
    def slots(self) -> int:
        return self.num_slots if self.num_slots else self.B + 1


WORKLOADS = {
    "C0": Workload("tiny-fp32", B=1, H=2, HV=2, K=32, V=32, T=4, L=8, io_dtype=FP32,
                   prefix=16, rounds=6),
    "C1": Workload("qwen3next-gdn-b1", B=1, H=16, HV=32, K=128, V=128, T=4, L=64,
                   prefix=64, rounds=200),
    "C2": Workload("qwen3next-gdn-sweep", B=128, H=16, HV=32, K=128, V=128, T=4, L=64,
                   num_slots=512, prefix=64, extra={"batches": [8, 32, 128, 256]}),
    "C3": Workload("qwen3next-gdn-flush-heavy", B=16, H=16, HV=32, K=128, V=128, T=4,
                   L=16, prefix=64, extra={"committed_tokens": 16384, "log_every": 512}),
    "C4": Workload("qwen3next-kda", B=64, H=16, HV=32, K=128, V=128, T=4, L=64,
                   per_key_gate=True, prefix=64, rounds=200, extra={"batches": [1, 64]}),
}


# ------------------------------------------------------------ draws

def rng_for(seed: int, *stream) -> np.random.Generator:
    """One independent PCG64 stream per (seed, stream labels)."""
    ss = np.random.SeedSequence([seed] + [zlib.crc32(s.encode()) if isinstance(s, str)
                                          else int(s) for s in stream])
    return np.random.Generator(np.random.PCG64(ss))


def layer_params(rng: np.random.Generator, HV: int, K: int, per_key_gate: bool):
    """A_log ~ U(0, ln 16) per v-head; dt_bias ~ U(-1, 1) per v-head (KDA: per channel)."""
    A_log = rng.uniform(0.0, math.log(16.0), size=HV).astype(np.float32)
    shape = (HV, K) if per_key_gate else (HV,)
    dt_bias = rng.uniform(-1.0, 1.0, size=shape).astype(np.float32)
    return A_log, dt_bias


def _row_scales(rng: np.random.Generator, shape, scale_range):
    """Per-row factors drawn log-uniformly from scale_range (lo, hi), shape + (1,)."""
    lo, hi = scale_range
    f = np.exp(rng.uniform(np.log(lo), np.log(hi), size=shape))
    return f.astype(np.float32)[..., None]


def window_inputs(rng: np.random.Generator, B: int, T: int, H: int, HV: int, K: int, V: int,
                  io_dtype: str, per_key_gate: bool = False, key_scale=None):
    """q, k, v, a, b ~ N(0, 1) with q, k scaled to unit norm per (token, head).
    key_scale=(lo, hi): q and k rows are then multiplied by factors drawn
    log-uniformly from [lo, hi] (raw, non-unit inputs)."""
    q = _unit_rows(rng.standard_normal((B, T, H, K), dtype=np.float32))
    k = _unit_rows(rng.standard_normal((B, T, H, K), dtype=np.float32))
    if key_scale is not None:
        q = q * _row_scales(rng, (B, T, H), key_scale)
        k = k * _row_scales(rng, (B, T, H), key_scale)
    v = rng.standard_normal((B, T, HV, V), dtype=np.float32)
    a_shape = (B, T, HV, K) if per_key_gate else (B, T, HV)
    a = rng.standard_normal(a_shape, dtype=np.float32)
    b = rng.standard_normal((B, T, HV), dtype=np.float32)
    return {name: store(x, io_dtype) for name, x in
            (("q", q), ("k", k), ("v", v), ("a", a), ("b", b))}


def token_stream(rng: np.random.Generator, n: int, H: int, HV: int, K: int, V: int,
                 io_dtype: str, per_key_gate: bool = False, key_scale=None):
    """Raw per-token records for a run of n tokens of one batch row:
    k [n, H, K] (unit norm; with key_scale=(lo, hi) each row then multiplied by a
    factor drawn log-uniformly from [lo, hi]), v [n, HV, V], a [n, HV] (KDA
    [n, HV, K]), b [n, HV]."""
    k = _unit_rows(rng.standard_normal((n, H, K), dtype=np.float32))
    if key_scale is not None:
        k = k * _row_scales(rng, (n, H), key_scale)
    v = rng.standard_normal((n, HV, V), dtype=np.float32)
    a = rng.standard_normal((n, HV, K) if per_key_gate else (n, HV), dtype=np.float32)
    b = rng.standard_normal((n, HV), dtype=np.float32)
    return {"k": store(k, io_dtype), "v": store(v, io_dtype), "a": a, "b": b}


def accept_lens(rng: np.random.Generator, B: int, T: int, full_frac: float = 0.0):
    """accept_len ~ U{1..T}; with full_frac > 0 that share of rows accepts all T."""
    acc = rng.integers(1, T + 1, size=B).astype(np.int32)
    if full_frac > 0:
        full = rng.random(B) < full_frac
        acc[full] = T
    return acc


def garbage_ring(rng: np.random.Generator, num_slots: int, H: int, HV: int, L: int, K: int,
                 V: int, io_dtype: str, per_key_gate: bool = False):
    """A random template for every ring array (a full-tensor compare against a copy
    of it catches writes to the wrong slot, position or head)."""
    gshape = (num_slots, HV, L, K) if per_key_gate else (num_slots, HV, L)
    return {
        "rawv": store(rng.standard_normal((num_slots, HV, L, V), dtype=np.float32), io_dtype),
        "rawk": store(rng.standard_normal((num_slots, H, L, K), dtype=np.float32), io_dtype),
        "g": rng.standard_normal(gshape, dtype=np.float32),
        "beta": rng.standard_normal((num_slots, HV, L), dtype=np.float32),
    }


def scattered_slots(rng: np.random.Generator, num_slots: int, B: int) -> np.ndarray:
    """B distinct slots drawn from a pool of num_slots (a random permutation prefix)."""
    return rng.permutation(num_slots)[:B].astype(np.int32)


def random_cursors(rng: np.random.Generator, num_slots: int, L: int, T: int):
    """Per-slot cache_base ~ U[0, L), write_pos ~ U[0, L - 2T], is_flush = 0."""
    base = rng.integers(0, L, size=num_slots).astype(np.int32)
    wp = rng.integers(0, L - 2 * T + 1, size=num_slots).astype(np.int32)
    return wp, base, np.zeros(num_slots, np.int32)
