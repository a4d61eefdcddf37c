"""fp64 CPU oracle for ReplaySSM ring spec-verify of one Gated DeltaNet layer.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The product library
(``gated_delta_rule_spec_gb300``) never imports it, and the two share no code:
this package wraps ``gdn_oracle.c`` (plain C, fp64, sequential), built with gcc
into ``oracle/_build/libgdn_oracle.so``.

Every array here is fp64 in the same index order as the device layout:

* checkpoint ``[num_slots, HV, V, K]``; ring ``rawv [num_slots, HV, L, V]``,
  ``rawk [num_slots, H, L, K]``, ``g [num_slots, HV, L]`` (KDA: ``[..., L, K]``),
  ``beta [num_slots, HV, L]``; cursors ``int32 [num_slots]``.
* window inputs ``q, k [B, T, H, K]``, ``v [B, T, HV, V]``, ``a, b [B, T, HV]``
  (KDA ``a [B, T, HV, K]``), ``A_log [HV]``, ``dt_bias [HV]`` (KDA ``[HV, K]``).

The method is the GDN recurrence ``S_t = exp(g_t) S_{t-1} (I - b_t k_t k_t^T) +
b_t v_t k_t^T``, ``o_t = S_t q_t`` with L2-normalised q, k (sglang PR #28695
"GDN ReplaySSM Ring Spec-Verify" and the blog post explaining it, §12.1), run
token by token in fp64.  Parity of every function is pinned against something
other than the oracle itself: verify, commit, fold and reset in
``tests/test_oracle_pins.py`` and ``tests/test_cursor_protocol.py``, prefill in
``tests/test_oracle_prefill_pins.py``, the snapshot comparison in
``tests/test_oracle_snapshot_pins.py``, the window's corrected deltas
(``verify_d``) in ``tests/test_oracle_derived_d_pins.py``; planted mistakes that the pins must catch
are in ``tests/test_oracle_mutations.py``.  None is marked "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdn_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libgdn_oracle.so")

ST_ACCEPT_RANGE = 1
ST_SLOT_OOR = 2
ST_RING_OVERFLOW = 4
ST_CURSOR_CORRUPT = 8
ST_UNFOLDED = 32

_lib = None


def build(force: bool = False) -> str:
    """Compile gdn_oracle.c with gcc (portable flags: no -march, no fast-math)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-std=c99", "-O2", "-fPIC", "-shared", "-fno-fast-math",
           "-ffp-contract=off", "-pthread", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class _Dims(ctypes.Structure):
    _fields_ = [("H", ctypes.c_int), ("HV", ctypes.c_int), ("K", ctypes.c_int),
                ("V", ctypes.c_int), ("T", ctypes.c_int), ("L", ctypes.c_int),
                ("num_slots", ctypes.c_int), ("per_key_gate", ctypes.c_int),
                ("scale", ctypes.c_double), ("l2_eps", ctypes.c_double)]


class _Layer(ctypes.Structure):
    _fields_ = [("checkpoint", ctypes.c_void_p), ("rawv", ctypes.c_void_p),
                ("rawk", ctypes.c_void_p), ("ring_g", ctypes.c_void_p),
                ("ring_beta", ctypes.c_void_p)]


class _Cursors(ctypes.Structure):
    _fields_ = [("write_pos", ctypes.c_void_p), ("cache_base", ctypes.c_void_p),
                ("is_flush", ctypes.c_void_p)]


def use_library(path: str | None) -> None:
    """Point the wrappers at another build of gdn_oracle.c (the mutation tests
    load deliberately broken copies); None returns to the normal build."""
    global _lib
    _lib = None
    _load(path)


def _load(path: str | None = None):
    global _lib
    if _lib is None:
        _lib = ctypes.CDLL(path or build())
        P = ctypes.c_void_p
        _lib.orc_softplus.restype = ctypes.c_double
        _lib.orc_softplus.argtypes = [ctypes.c_double]
        _lib.orc_gate_g.restype = ctypes.c_double
        _lib.orc_gate_g.argtypes = [ctypes.c_double] * 3
        _lib.orc_gate_beta.restype = ctypes.c_double
        _lib.orc_gate_beta.argtypes = [ctypes.c_double]
        _lib.orc_step.restype = None
        _lib.orc_step.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, P, P, P, P,
                                  ctypes.c_double, ctypes.c_double]
        _lib.orc_readout.restype = None
        _lib.orc_readout.argtypes = [ctypes.c_int, ctypes.c_int, P, P, ctypes.c_double,
                                     ctypes.c_double, P]
        _lib.orc_verify.restype = ctypes.c_uint32
        _lib.orc_verify.argtypes = [P, P, P, P, ctypes.c_int] + [P] * 8 + [P, ctypes.c_int]
        _lib.orc_verify_d.restype = ctypes.c_uint32
        _lib.orc_verify_d.argtypes = [P, P, P, P, ctypes.c_int] + [P] * 8 + [P, ctypes.c_int]
        _lib.orc_commit.restype = ctypes.c_uint32
        _lib.orc_commit.argtypes = [P, P, P, ctypes.c_int, P]
        _lib.orc_fold.restype = ctypes.c_uint32
        _lib.orc_fold.argtypes = [P, P, ctypes.c_int, P, P, ctypes.c_int, ctypes.c_int]
        _lib.orc_reset.restype = ctypes.c_uint32
        _lib.orc_reset.argtypes = [P, P, P, ctypes.c_int]
        _lib.orc_prefill.restype = ctypes.c_uint32
        _lib.orc_prefill.argtypes = [P, P, P, P, ctypes.c_int, ctypes.c_int] + [P] * 8 + [
            ctypes.c_int, ctypes.c_int]
        _lib.orc_snapshot_verify.restype = ctypes.c_uint32
        _lib.orc_snapshot_verify.argtypes = [P, P, P, ctypes.c_int] + [P] * 9
        _lib.orc_snapshot_commit.restype = ctypes.c_uint32
        _lib.orc_snapshot_commit.argtypes = [P, P, P, ctypes.c_int, P, P]
        _lib.orc_run.restype = None
        _lib.orc_run.argtypes = [P, P, ctypes.c_int, P, P, P, P]
        _lib.orc_run_batch.restype = None
        _lib.orc_run_batch.argtypes = [P, ctypes.c_int, P, ctypes.c_int, P, P, P, P, ctypes.c_int]
    return _lib


def _f64(x) -> np.ndarray:
    a = np.ascontiguousarray(x, dtype=np.float64)
    return a


def _i32(x) -> np.ndarray:
    return np.ascontiguousarray(x, dtype=np.int32)


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


@dataclass
class Dims:
    H: int
    HV: int
    K: int
    V: int
    T: int
    L: int
    num_slots: int
    per_key_gate: bool = False
    scale: float = 1.0
    l2_eps: float = 1e-6

    def _c(self) -> _Dims:
        return _Dims(self.H, self.HV, self.K, self.V, self.T, self.L, self.num_slots,
                     int(self.per_key_gate), float(self.scale), float(self.l2_eps))

    @property
    def gw(self) -> int:
        return self.K if self.per_key_gate else 1


class Layer:
    """fp64 layer state: checkpoint + raw ring.  Arrays are owned numpy fp64."""

    def __init__(self, dims: Dims, checkpoint=None, rawv=None, rawk=None, ring_g=None,
                 ring_beta=None):
        d = dims
        self.dims = d
        z = np.zeros
        self.checkpoint = _f64(checkpoint if checkpoint is not None
                               else z((d.num_slots, d.HV, d.V, d.K)))
        self.rawv = _f64(rawv if rawv is not None else z((d.num_slots, d.HV, d.L, d.V)))
        self.rawk = _f64(rawk if rawk is not None else z((d.num_slots, d.H, d.L, d.K)))
        gshape = (d.num_slots, d.HV, d.L) + ((d.K,) if d.per_key_gate else ())
        self.ring_g = _f64(ring_g if ring_g is not None else z(gshape))
        self.ring_beta = _f64(ring_beta if ring_beta is not None
                              else z((d.num_slots, d.HV, d.L)))

    def _c(self) -> _Layer:
        return _Layer(self.checkpoint.ctypes.data, self.rawv.ctypes.data,
                      self.rawk.ctypes.data, self.ring_g.ctypes.data,
                      self.ring_beta.ctypes.data)

    def copy(self) -> "Layer":
        return Layer(self.dims, self.checkpoint.copy(), self.rawv.copy(), self.rawk.copy(),
                     self.ring_g.copy(), self.ring_beta.copy())


class Cursors:
    def __init__(self, num_slots: int, write_pos=None, cache_base=None, is_flush=None):
        z = np.zeros(num_slots, np.int32)
        self.write_pos = _i32(write_pos if write_pos is not None else z)
        self.cache_base = _i32(cache_base if cache_base is not None else z.copy())
        self.is_flush = _i32(is_flush if is_flush is not None else z.copy())

    def _c(self) -> _Cursors:
        return _Cursors(self.write_pos.ctypes.data, self.cache_base.ctypes.data,
                        self.is_flush.ctypes.data)

    def copy(self) -> "Cursors":
        return Cursors(len(self.write_pos), self.write_pos.copy(), self.cache_base.copy(),
                       self.is_flush.copy())


# ---------------------------------------------------------------- scalar math

def softplus(x: float) -> float:
    return _load().orc_softplus(float(x))


def gate_g(A_log: float, a: float, dt_bias: float) -> float:
    return _load().orc_gate_g(float(A_log), float(a), float(dt_bias))


def gate_beta(b: float) -> float:
    return _load().orc_gate_beta(float(b))


def gate(A_log, a, dt_bias, b, per_key_gate: bool = False):
    """Vectorised gating over arrays (loops the scalar C functions).

    GDN: a, b [..., HV], A_log, dt_bias [HV].  KDA: a [..., HV, K], dt_bias [HV, K].
    Returns (g, beta) as fp64 arrays shaped like a and b.
    """
    lib = _load()
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    A_log = np.asarray(A_log, np.float64)
    dt_bias = np.asarray(dt_bias, np.float64)
    g = np.empty_like(a)
    if per_key_gate:
        HV, K = dt_bias.shape
        af = a.reshape(-1, HV, K)
        gf = g.reshape(-1, HV, K)
        for i in range(af.shape[0]):
            for hv in range(HV):
                for j in range(K):
                    gf[i, hv, j] = lib.orc_gate_g(A_log[hv], af[i, hv, j], dt_bias[hv, j])
    else:
        HV = dt_bias.shape[0]
        af = a.reshape(-1, HV)
        gf = g.reshape(-1, HV)
        for i in range(af.shape[0]):
            for hv in range(HV):
                gf[i, hv] = lib.orc_gate_g(A_log[hv], af[i, hv], dt_bias[hv])
    beta = np.vectorize(lib.orc_gate_beta, otypes=[np.float64])(b) if b.size else b.copy()
    return g, beta


# ---------------------------------------------------------------- recurrence

def step(S, v, k_raw, g, beta, eps: float = 1e-6, per_key_gate: bool = False):
    """One recurrence step on a copy of S [V, K]; returns the new state."""
    S = _f64(np.array(S, dtype=np.float64, copy=True))
    V, K = S.shape
    v = _f64(v)
    k_raw = _f64(k_raw)
    g = _f64(np.atleast_1d(g))
    _load().orc_step(V, K, int(per_key_gate), _ptr(S), _ptr(v), _ptr(k_raw), _ptr(g),
                     float(beta), float(eps))
    return S


def readout(S, q_raw, eps: float = 1e-6, scale: float = 1.0):
    S = _f64(S)
    V, K = S.shape
    q_raw = _f64(q_raw)
    o = np.empty(V, np.float64)
    _load().orc_readout(V, K, _ptr(S), _ptr(q_raw), float(eps), float(scale), _ptr(o))
    return o


def run(dims: Dims, S, v, k_raw, g, beta):
    """Recurrence over n tokens from S (returns a new array).  v [n,V], k [n,K],
    g [n] or [n,K], beta [n]."""
    S = _f64(np.array(S, dtype=np.float64, copy=True))
    v, k_raw, g, beta = _f64(v), _f64(k_raw), _f64(g), _f64(beta)
    n = v.shape[0]
    _load().orc_run(ctypes.byref(dims._c()), _ptr(S), n, _ptr(v), _ptr(k_raw), _ptr(g),
                    _ptr(beta))
    return S


def run_batch(dims: Dims, S, v, k_raw, g, beta, nthreads: int = 1):
    """Independent recurrences for many units at once (threads over units).
    S [U, V, K]; v [U, n, V]; k_raw [U, n, K]; g [U, n] or [U, n, K]; beta [U, n].
    Returns the new states [U, V, K]."""
    S = _f64(np.array(S, dtype=np.float64, copy=True))
    v, k_raw, g, beta = _f64(v), _f64(k_raw), _f64(g), _f64(beta)
    U, n = v.shape[0], v.shape[1]
    _load().orc_run_batch(ctypes.byref(dims._c()), U, _ptr(S), n, _ptr(v), _ptr(k_raw), _ptr(g),
                          _ptr(beta), int(nthreads))
    return S


# ---------------------------------------------------------------- layer calls

def verify(dims: Dims, layer: Layer, cursors: Cursors, slot_idx, q, k, v, a, b, A_log,
           dt_bias, unit_mask=None, nthreads: int = 1):
    """Verify one batch: returns (out [B,T,HV,V] fp64, status bits).  Writes the
    draft window's raw records into ``layer``'s ring (the side channel)."""
    slot_idx = _i32(slot_idx)
    B = slot_idx.shape[0]
    q, k, v, a, b = _f64(q), _f64(k), _f64(v), _f64(a), _f64(b)
    A_log, dt_bias = _f64(A_log), _f64(dt_bias)
    out = np.zeros((B, dims.T, dims.HV, dims.V), np.float64)
    mask = None if unit_mask is None else np.ascontiguousarray(unit_mask, np.uint8)
    cd, cl, cc = dims._c(), layer._c(), cursors._c()
    st = _load().orc_verify(ctypes.byref(cd), ctypes.byref(cl), ctypes.byref(cc),
                            _ptr(slot_idx), B, _ptr(q), _ptr(k), _ptr(v), _ptr(a), _ptr(b),
                            _ptr(A_log), _ptr(dt_bias), _ptr(out), _ptr(mask), int(nthreads))
    return out, int(st)


def verify_d(dims: Dims, layer: Layer, cursors: Cursors, slot_idx, q, k, v, a, b, A_log,
             dt_bias, nthreads: int = 1):
    """verify() that also returns the corrected delta of every window token:
    (out [B,T,HV,V], d [B,T,HV,V], status bits), with d_t = beta_t (v_t - S k^_t)
    taken against the decayed state before token t (blog post on sglang PR
    #28695, §12.1).  These are what a ring caching d instead of raw v (the
    derived-d design) would hold for the window's records."""
    slot_idx = _i32(slot_idx)
    B = slot_idx.shape[0]
    q, k, v, a, b = _f64(q), _f64(k), _f64(v), _f64(a), _f64(b)
    A_log, dt_bias = _f64(A_log), _f64(dt_bias)
    out = np.zeros((B, dims.T, dims.HV, dims.V), np.float64)
    dwin = np.zeros((B, dims.T, dims.HV, dims.V), np.float64)
    cd, cl, cc = dims._c(), layer._c(), cursors._c()
    st = _load().orc_verify_d(ctypes.byref(cd), ctypes.byref(cl), ctypes.byref(cc),
                              _ptr(slot_idx), B, _ptr(q), _ptr(k), _ptr(v), _ptr(a), _ptr(b),
                              _ptr(A_log), _ptr(dt_bias), _ptr(out), _ptr(dwin), int(nthreads))
    return out, dwin, int(st)


def commit(dims: Dims, cursors: Cursors, slot_idx, accept_len) -> int:
    slot_idx, accept_len = _i32(slot_idx), _i32(accept_len)
    cd, cc = dims._c(), cursors._c()
    return int(_load().orc_commit(ctypes.byref(cd), ctypes.byref(cc), _ptr(slot_idx),
                                  slot_idx.shape[0], _ptr(accept_len)))


def fold(dims: Dims, layers, cursors: Cursors, slot_idx, nthreads: int = 1) -> int:
    if isinstance(layers, Layer):
        layers = [layers]
    slot_idx = _i32(slot_idx)
    arr = (_Layer * len(layers))(*[ly._c() for ly in layers])
    cd, cc = dims._c(), cursors._c()
    return int(_load().orc_fold(ctypes.byref(cd), arr, len(layers), ctypes.byref(cc),
                                _ptr(slot_idx), slot_idx.shape[0], int(nthreads)))


def prefill(dims: Dims, layer: Layer, cursors: Cursors, slot_idx, q, k, v, a, b, A_log, dt_bias,
            from_zero: bool = True, nthreads: int = 1):
    """Prefill of N prompt tokens per row: returns (out [B, N, HV, V] fp64, status
    bits).  The final states replace the rows' checkpoints and the rows' cursors
    are reset.  q, k [B, N, H, K]; v [B, N, HV, V]; a, b [B, N, HV] (KDA a
    [B, N, HV, K]).  ``from_zero=False`` continues from the checkpoint and needs
    an empty ring (write_pos 0), else the row is skipped with ST_UNFOLDED."""
    slot_idx = _i32(slot_idx)
    B = slot_idx.shape[0]
    q, k, v, a, b = _f64(q), _f64(k), _f64(v), _f64(a), _f64(b)
    A_log, dt_bias = _f64(A_log), _f64(dt_bias)
    N = q.shape[1]
    out = np.zeros((B, N, dims.HV, dims.V), np.float64)
    cd, cl, cc = dims._c(), layer._c(), cursors._c()
    st = _load().orc_prefill(ctypes.byref(cd), ctypes.byref(cl), ctypes.byref(cc), _ptr(slot_idx),
                             B, N, _ptr(q), _ptr(k), _ptr(v), _ptr(a), _ptr(b), _ptr(A_log),
                             _ptr(dt_bias), _ptr(out), int(bool(from_zero)), int(nthreads))
    return out, int(st)


def snapshot_verify(dims: Dims, layer: Layer, slot_idx, q, k, v, a, b, A_log, dt_bias):
    """Comparison variant (the per-draft snapshot design the ring replaces):
    returns (out [B,T,HV,V], snapshots [B,T,HV,V,K], status bits); the state
    after each window token is stored, the checkpoint is only read."""
    slot_idx = _i32(slot_idx)
    B = slot_idx.shape[0]
    q, k, v, a, b = _f64(q), _f64(k), _f64(v), _f64(a), _f64(b)
    A_log, dt_bias = _f64(A_log), _f64(dt_bias)
    out = np.zeros((B, dims.T, dims.HV, dims.V), np.float64)
    snap = np.zeros((B, dims.T, dims.HV, dims.V, dims.K), np.float64)
    cd, cl = dims._c(), layer._c()
    st = _load().orc_snapshot_verify(ctypes.byref(cd), ctypes.byref(cl), _ptr(slot_idx), B, _ptr(q),
                                     _ptr(k), _ptr(v), _ptr(a), _ptr(b), _ptr(A_log), _ptr(dt_bias),
                                     _ptr(out), _ptr(snap))
    return out, snap, int(st)


def snapshot_commit(dims: Dims, layer: Layer, slot_idx, accept_len, snap) -> int:
    """Comparison variant: checkpoint[slot] = snap[b, accept_len - 1]."""
    slot_idx, accept_len = _i32(slot_idx), _i32(accept_len)
    snap = _f64(snap)
    cd, cl = dims._c(), layer._c()
    return int(_load().orc_snapshot_commit(ctypes.byref(cd), ctypes.byref(cl), _ptr(slot_idx),
                                           slot_idx.shape[0], _ptr(accept_len), _ptr(snap)))


def reset(dims: Dims, cursors: Cursors, slot_idx) -> int:
    slot_idx = _i32(slot_idx)
    cd, cc = dims._c(), cursors._c()
    return int(_load().orc_reset(ctypes.byref(cd), ctypes.byref(cc), _ptr(slot_idx),
                                 slot_idx.shape[0]))
