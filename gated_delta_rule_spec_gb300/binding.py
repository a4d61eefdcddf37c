"""Python binding of libgdnspec (include/gdn_spec.h): argument marshalling only.

Every step of the path runs in the library's CUDA kernels.  PyTorch supplies
device memory and streams; tensors are passed as raw device pointers.  If the
library has not been built, the first call raises with the build command; there
is no fallback of any kind.

Names follow the C ABI: ``verify``, ``commit``, ``fold``, ``reset``,
``read_status`` wrap ``gdn_spec_verify`` ... ``gdn_spec_read_status``.
``SpecLayer`` and ``SpecCursors`` allocate the per-layer state and the shared
cursors with torch and produce the C descriptors.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

GATE_SCALAR, GATE_PER_KEY = 0, 1
DTYPE_BF16, DTYPE_FP32 = 0, 1
ST_ACCEPT_RANGE, ST_SLOT_OOR, ST_RING_OVERFLOW, ST_CURSOR_CORRUPT, ST_TIMEOUT = 1, 2, 4, 8, 16
ST_UNFOLDED = 32

_IO_TORCH = {DTYPE_BF16: torch.bfloat16, DTYPE_FP32: torch.float32}
_NAME_TO_DTYPE = {"bf16": DTYPE_BF16, "fp32": DTYPE_FP32}


class GdnSpecError(RuntimeError):
    pass


class LayerDesc(ctypes.Structure):
    _fields_ = [("H", ctypes.c_int32), ("HV", ctypes.c_int32), ("K", ctypes.c_int32),
                ("V", ctypes.c_int32), ("T", ctypes.c_int32), ("L", ctypes.c_int32),
                ("num_slots", ctypes.c_int32), ("gate_kind", ctypes.c_int32),
                ("io_dtype", ctypes.c_int32), ("scale", ctypes.c_float),
                ("l2_eps", ctypes.c_float), ("checkpoint", ctypes.c_void_p),
                ("rawv", ctypes.c_void_p), ("rawk", ctypes.c_void_p),
                ("ring_g", ctypes.c_void_p), ("ring_beta", ctypes.c_void_p)]


class CursorDesc(ctypes.Structure):
    _fields_ = [("num_slots", ctypes.c_int32), ("write_pos", ctypes.c_void_p),
                ("cache_base", ctypes.c_void_p), ("is_flush", ctypes.c_void_p),
                ("status", ctypes.c_void_p)]


_lib = None
EXPORTS = ("gdn_spec_verify", "gdn_spec_verify_d", "gdn_spec_commit", "gdn_spec_fold",
           "gdn_spec_reset", "gdn_spec_prefill",
           "gdn_spec_snapshot_verify", "gdn_spec_snapshot_commit",
           "gdn_spec_read_status", "gdn_spec_strerror", "gdn_spec_abi_version",
           "gdn_spec_verify_path", "gdn_spec_prefill_path", "gdn_spec_set_wait_limit")


def library_path() -> str:
    return _build.LIB


def load() -> ctypes.CDLL:
    """Load libgdnspec.so (built in-tree).  Raises if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    path = library_path()
    if not os.path.exists(path):
        raise GdnSpecError(
            f"libgdnspec.so not found at {path}; build it with "
            "`python -c 'import __graft_entry__ as g; g.build()'`")
    lib = ctypes.CDLL(path)
    P, I32 = ctypes.c_void_p, ctypes.c_int32
    LP, CP = ctypes.POINTER(LayerDesc), ctypes.POINTER(CursorDesc)
    lib.gdn_spec_verify.argtypes = [LP, CP, P, I32, P, P, P, P, P, P, P, P, P]
    lib.gdn_spec_verify_d.argtypes = [LP, P, CP, P, I32, P, P, P, P, P, P, P, P, P]
    lib.gdn_spec_commit.argtypes = [CP, I32, I32, P, I32, P, P]
    lib.gdn_spec_fold.argtypes = [LP, I32, CP, P, I32, P]
    lib.gdn_spec_reset.argtypes = [CP, P, I32, P]
    lib.gdn_spec_prefill.argtypes = [LP, CP, P, I32, I32, P, P, P, P, P, P, P, P, I32, P]
    lib.gdn_spec_snapshot_verify.argtypes = [LP, CP, P, I32, P, P, P, P, P, P, P, P, P, P]
    lib.gdn_spec_snapshot_commit.argtypes = [LP, CP, P, I32, P, P, P]
    lib.gdn_spec_read_status.argtypes = [CP, ctypes.POINTER(ctypes.c_uint32), I32, P]
    for name in ("gdn_spec_verify", "gdn_spec_verify_d", "gdn_spec_commit", "gdn_spec_fold",
                 "gdn_spec_reset",
                 "gdn_spec_prefill", "gdn_spec_snapshot_verify", "gdn_spec_snapshot_commit",
                 "gdn_spec_read_status"):
        getattr(lib, name).restype = ctypes.c_int
    lib.gdn_spec_strerror.argtypes = [ctypes.c_int]
    lib.gdn_spec_strerror.restype = ctypes.c_char_p
    lib.gdn_spec_abi_version.argtypes = []
    lib.gdn_spec_abi_version.restype = ctypes.c_int
    lib.gdn_spec_verify_path.argtypes = [LP]
    lib.gdn_spec_verify_path.restype = ctypes.c_char_p
    lib.gdn_spec_prefill_path.argtypes = [LP]
    lib.gdn_spec_prefill_path.restype = ctypes.c_char_p
    lib.gdn_spec_set_wait_limit.argtypes = [ctypes.c_uint32]
    lib.gdn_spec_set_wait_limit.restype = ctypes.c_uint32
    _lib = lib
    return lib


def _check(rc: int, what: str) -> None:
    if rc != 0:
        raise GdnSpecError(f"{what}: {load().gdn_spec_strerror(rc).decode()} (code {rc})")


def _ptr(t: torch.Tensor | None):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _need(t: torch.Tensor, name: str, dtype: torch.dtype, shape: tuple) -> None:
    if t.dtype != dtype or tuple(t.shape) != tuple(shape) or not t.is_contiguous() or not t.is_cuda:
        raise GdnSpecError(f"{name}: want contiguous CUDA {dtype} {tuple(shape)}, got "
                           f"{t.dtype} {tuple(t.shape)} contiguous={t.is_contiguous()} "
                           f"device={t.device}")


class SpecCursors:
    """Per-slot cursors (shared by all layers) and the device status word."""

    def __init__(self, num_slots: int, device="cuda"):
        self.num_slots = num_slots
        z = lambda: torch.zeros(num_slots, dtype=torch.int32, device=device)  # noqa: E731
        self.write_pos, self.cache_base, self.is_flush = z(), z(), z()
        self.status = torch.zeros(4, dtype=torch.int32, device=device)  # word 0 is used

    def desc(self) -> CursorDesc:
        return CursorDesc(self.num_slots, self.write_pos.data_ptr(), self.cache_base.data_ptr(),
                          self.is_flush.data_ptr(), self.status.data_ptr())


class SpecLayer:
    """One GDN layer's dimensions and per-slot state (checkpoint + raw ring)."""

    def __init__(self, H: int, HV: int, K: int, V: int, T: int, L: int, num_slots: int,
                 per_key_gate: bool = False, io_dtype: str = "bf16", scale: float = 1.0,
                 l2_eps: float = 1e-6, device="cuda"):
        self.H, self.HV, self.K, self.V, self.T, self.L = H, HV, K, V, T, L
        self.num_slots = num_slots
        self.per_key_gate = per_key_gate
        self.io_code = _NAME_TO_DTYPE[io_dtype]
        self.io_torch = _IO_TORCH[self.io_code]
        self.scale, self.l2_eps = scale, l2_eps
        f32 = torch.float32
        self.checkpoint = torch.zeros(num_slots, HV, V, K, dtype=f32, device=device)
        self.rawv = torch.zeros(num_slots, HV, L, V, dtype=self.io_torch, device=device)
        self.rawk = torch.zeros(num_slots, H, L, K, dtype=self.io_torch, device=device)
        gshape = (num_slots, HV, L, K) if per_key_gate else (num_slots, HV, L)
        self.ring_g = torch.zeros(gshape, dtype=f32, device=device)
        self.ring_beta = torch.zeros(num_slots, HV, L, dtype=f32, device=device)

    def desc(self) -> LayerDesc:
        return LayerDesc(self.H, self.HV, self.K, self.V, self.T, self.L, self.num_slots,
                         GATE_PER_KEY if self.per_key_gate else GATE_SCALAR, self.io_code,
                         self.scale, self.l2_eps, self.checkpoint.data_ptr(),
                         self.rawv.data_ptr(), self.rawk.data_ptr(), self.ring_g.data_ptr(),
                         self.ring_beta.data_ptr())

    def new_dring(self) -> torch.Tensor:
        """A zeroed d ring for gdn_spec_verify_d: fp32 [num_slots, HV, L, V]."""
        return torch.zeros(self.num_slots, self.HV, self.L, self.V, dtype=torch.float32,
                           device=self.checkpoint.device)

    def window_shapes(self, B: int) -> dict:
        T, H, HV, K, V = self.T, self.H, self.HV, self.K, self.V
        return {"q": (B, T, H, K), "k": (B, T, H, K), "v": (B, T, HV, V),
                "a": (B, T, HV, K) if self.per_key_gate else (B, T, HV), "b": (B, T, HV),
                "A_log": (HV,), "dt_bias": (HV, K) if self.per_key_gate else (HV,),
                "out": (B, T, HV, V)}


def verify_path(layer: SpecLayer) -> str:
    r = load().gdn_spec_verify_path(ctypes.byref(layer.desc()))
    if r is None:
        raise GdnSpecError("invalid layer descriptor")
    return r.decode()


def prefill_path(layer: SpecLayer) -> str:
    r = load().gdn_spec_prefill_path(ctypes.byref(layer.desc()))
    if r is None:
        raise GdnSpecError("invalid layer descriptor")
    return r.decode()


def verify(layer: SpecLayer, cursors: SpecCursors, slot_idx: torch.Tensor, q, k, v, a, b,
           A_log, dt_bias, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """gdn_spec_verify: outputs of the draft window [B, T, HV, V]; writes the ring."""
    B = slot_idx.shape[0]
    shp = layer.window_shapes(B)
    io = layer.io_torch
    _need(slot_idx, "slot_idx", torch.int32, (B,))
    for name, t in (("q", q), ("k", k), ("v", v), ("a", a), ("b", b)):
        _need(t, name, io, shp[name])
    _need(A_log, "A_log", torch.float32, shp["A_log"])
    _need(dt_bias, "dt_bias", torch.float32, shp["dt_bias"])
    if out is None:
        out = torch.empty(shp["out"], dtype=io, device=q.device)
    _need(out, "out", io, shp["out"])
    rc = load().gdn_spec_verify(ctypes.byref(layer.desc()), ctypes.byref(cursors.desc()),
                                _ptr(slot_idx), B, _ptr(q), _ptr(k), _ptr(v), _ptr(a), _ptr(b),
                                _ptr(A_log), _ptr(dt_bias), _ptr(out), _stream(stream))
    _check(rc, "gdn_spec_verify")
    return out


def verify_d(layer: SpecLayer, dring: torch.Tensor, cursors: SpecCursors, slot_idx: torch.Tensor,
             q, k, v, a, b, A_log, dt_bias, out: torch.Tensor | None = None,
             stream=None) -> torch.Tensor:
    """gdn_spec_verify_d (comparison variant): outputs of the draft window
    [B, T, HV, V] from a ring that also caches each token's corrected delta;
    writes the window's raw records into the ring and its d into ``dring``
    (fp32 [num_slots, HV, L, V], see ``SpecLayer.new_dring``)."""
    B = slot_idx.shape[0]
    shp = layer.window_shapes(B)
    io = layer.io_torch
    _need(slot_idx, "slot_idx", torch.int32, (B,))
    for name, t in (("q", q), ("k", k), ("v", v), ("a", a), ("b", b)):
        _need(t, name, io, shp[name])
    _need(A_log, "A_log", torch.float32, shp["A_log"])
    _need(dt_bias, "dt_bias", torch.float32, shp["dt_bias"])
    _need(dring, "dring", torch.float32, (layer.num_slots, layer.HV, layer.L, layer.V))
    if out is None:
        out = torch.empty(shp["out"], dtype=io, device=q.device)
    _need(out, "out", io, shp["out"])
    rc = load().gdn_spec_verify_d(ctypes.byref(layer.desc()), _ptr(dring), ctypes.byref(cursors.desc()),
                                  _ptr(slot_idx), B, _ptr(q), _ptr(k), _ptr(v), _ptr(a), _ptr(b),
                                  _ptr(A_log), _ptr(dt_bias), _ptr(out), _stream(stream))
    _check(rc, "gdn_spec_verify_d")
    return out


def commit(cursors: SpecCursors, T: int, L: int, slot_idx: torch.Tensor,
           accept_len: torch.Tensor, stream=None) -> None:
    B = slot_idx.shape[0]
    _need(slot_idx, "slot_idx", torch.int32, (B,))
    _need(accept_len, "accept_len", torch.int32, (B,))
    rc = load().gdn_spec_commit(ctypes.byref(cursors.desc()), T, L, _ptr(slot_idx), B,
                                _ptr(accept_len), _stream(stream))
    _check(rc, "gdn_spec_commit")


def fold(layers, cursors: SpecCursors, slot_idx: torch.Tensor, stream=None) -> None:
    if isinstance(layers, SpecLayer):
        layers = [layers]
    B = slot_idx.shape[0]
    _need(slot_idx, "slot_idx", torch.int32, (B,))
    arr = (LayerDesc * len(layers))(*[ly.desc() for ly in layers])
    rc = load().gdn_spec_fold(arr, len(layers), ctypes.byref(cursors.desc()), _ptr(slot_idx), B,
                              _stream(stream))
    _check(rc, "gdn_spec_fold")


def prefill(layer: SpecLayer, cursors: SpecCursors, slot_idx: torch.Tensor, q, k, v, a, b,
            A_log, dt_bias, out: torch.Tensor | None = None, from_zero: bool = True,
            stream=None) -> torch.Tensor:
    """gdn_spec_prefill: outputs of the N prompt tokens [B, N, HV, V]; the final
    states become the slots' checkpoints and the slots' cursors are reset."""
    B = slot_idx.shape[0]
    N = q.shape[1]
    T, H, HV, K, V = N, layer.H, layer.HV, layer.K, layer.V
    io = layer.io_torch
    _need(slot_idx, "slot_idx", torch.int32, (B,))
    shp = {"q": (B, T, H, K), "k": (B, T, H, K), "v": (B, T, HV, V),
           "a": (B, T, HV, K) if layer.per_key_gate else (B, T, HV), "b": (B, T, HV)}
    for name, t in (("q", q), ("k", k), ("v", v), ("a", a), ("b", b)):
        _need(t, name, io, shp[name])
    _need(A_log, "A_log", torch.float32, (HV,))
    _need(dt_bias, "dt_bias", torch.float32, (HV, K) if layer.per_key_gate else (HV,))
    if out is None:
        out = torch.empty((B, N, HV, V), dtype=io, device=q.device)
    _need(out, "out", io, (B, N, HV, V))
    rc = load().gdn_spec_prefill(ctypes.byref(layer.desc()), ctypes.byref(cursors.desc()),
                                 _ptr(slot_idx), B, N, _ptr(q), _ptr(k), _ptr(v), _ptr(a), _ptr(b),
                                 _ptr(A_log), _ptr(dt_bias), _ptr(out), int(bool(from_zero)),
                                 _stream(stream))
    _check(rc, "gdn_spec_prefill")
    return out


def snapshot_verify(layer: SpecLayer, cursors: SpecCursors, slot_idx: torch.Tensor, q, k, v, a, b,
                    A_log, dt_bias, out: torch.Tensor | None = None,
                    snap: torch.Tensor | None = None, stream=None):
    """Comparison variant (per-draft snapshots): returns (out [B, T, HV, V],
    snap fp32 [B, T, HV, V, K]); the checkpoint is only read."""
    B = slot_idx.shape[0]
    shp = layer.window_shapes(B)
    io = layer.io_torch
    _need(slot_idx, "slot_idx", torch.int32, (B,))
    for name, t in (("q", q), ("k", k), ("v", v), ("a", a), ("b", b)):
        _need(t, name, io, shp[name])
    _need(A_log, "A_log", torch.float32, shp["A_log"])
    _need(dt_bias, "dt_bias", torch.float32, shp["dt_bias"])
    if out is None:
        out = torch.empty(shp["out"], dtype=io, device=q.device)
    _need(out, "out", io, shp["out"])
    sshape = (B, layer.T, layer.HV, layer.V, layer.K)
    if snap is None:
        snap = torch.empty(sshape, dtype=torch.float32, device=q.device)
    _need(snap, "snap", torch.float32, sshape)
    rc = load().gdn_spec_snapshot_verify(ctypes.byref(layer.desc()), ctypes.byref(cursors.desc()),
                                         _ptr(slot_idx), B, _ptr(q), _ptr(k), _ptr(v), _ptr(a),
                                         _ptr(b), _ptr(A_log), _ptr(dt_bias), _ptr(out), _ptr(snap),
                                         _stream(stream))
    _check(rc, "gdn_spec_snapshot_verify")
    return out, snap


def snapshot_commit(layer: SpecLayer, cursors: SpecCursors, slot_idx: torch.Tensor,
                    accept_len: torch.Tensor, snap: torch.Tensor, stream=None) -> None:
    """Comparison variant: checkpoint[slot] = snap[b, accept_len - 1]."""
    B = slot_idx.shape[0]
    _need(slot_idx, "slot_idx", torch.int32, (B,))
    _need(accept_len, "accept_len", torch.int32, (B,))
    _need(snap, "snap", torch.float32, (B, layer.T, layer.HV, layer.V, layer.K))
    rc = load().gdn_spec_snapshot_commit(ctypes.byref(layer.desc()), ctypes.byref(cursors.desc()),
                                         _ptr(slot_idx), B, _ptr(accept_len), _ptr(snap),
                                         _stream(stream))
    _check(rc, "gdn_spec_snapshot_commit")


def reset(cursors: SpecCursors, slot_idx: torch.Tensor, stream=None) -> None:
    B = slot_idx.shape[0]
    _need(slot_idx, "slot_idx", torch.int32, (B,))
    rc = load().gdn_spec_reset(ctypes.byref(cursors.desc()), _ptr(slot_idx), B, _stream(stream))
    _check(rc, "gdn_spec_reset")


def read_status(cursors: SpecCursors, clear: bool = True, stream=None) -> int:
    v = ctypes.c_uint32(0)
    rc = load().gdn_spec_read_status(ctypes.byref(cursors.desc()), ctypes.byref(v), int(clear),
                                     _stream(stream))
    _check(rc, "gdn_spec_read_status")
    return int(v.value)


WAIT_LIMIT_DEFAULT = 0xFFFFFFFF


def set_wait_limit(polls: int) -> int:
    """gdn_spec_set_wait_limit (diagnostic): polls after which the first wait on
    each data copy gives up; WAIT_LIMIT_DEFAULT restores the default.  Returns
    the previous limit."""
    return int(load().gdn_spec_set_wait_limit(ctypes.c_uint32(polls & 0xFFFFFFFF)))
