"""Host-side argument checks of every C-ABI entry point, without a GPU.

Each entry point validates its descriptors and arguments before its first CUDA
call, and a batch of B = 0 returns before any launch.  So every case here either
fails validation or has B = 0, and the fake (aligned, never dereferenced) device
pointers are never used.  The expected codes are the ones include/gdn_spec.h
documents.
"""
import ctypes

import pytest

from gated_delta_rule_spec_gb300 import binding
from gated_delta_rule_spec_gb300 import build as lib_build

OK, EINVAL, EDTYPE, EALIGN, EUNSUP = 0, -1, -2, -3, -5
FAKE = 0x7F0000100000            # 16-byte aligned, never dereferenced
MIS = FAKE + 8                    # not 16-byte aligned


@pytest.fixture(scope="module")
def lib():
    lib_build.build()
    return binding.load()


def layer(**kw):
    f = dict(H=16, HV=32, K=128, V=128, T=4, L=64, num_slots=8, gate_kind=binding.GATE_SCALAR,
             io_dtype=binding.DTYPE_BF16, scale=1.0, l2_eps=1e-6, checkpoint=FAKE, rawv=FAKE,
             rawk=FAKE, ring_g=FAKE, ring_beta=FAKE)
    f.update(kw)
    return binding.LayerDesc(*(f[n] for n, _ in binding.LayerDesc._fields_))


def cursors(**kw):
    f = dict(num_slots=8, write_pos=FAKE, cache_base=FAKE, is_flush=FAKE, status=FAKE)
    f.update(kw)
    return binding.CursorDesc(*(f[n] for n, _ in binding.CursorDesc._fields_))


def _ref(x):
    return None if x is None else ctypes.byref(x)


def verify(lib, ly, cu, B=1, slot=FAKE, q=FAKE, out=FAKE):
    return lib.gdn_spec_verify(_ref(ly), _ref(cu), slot, B, q, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE,
                               out, None)


@pytest.mark.parametrize("kw,want", [
    (dict(HV=24), EINVAL),                         # H does not divide HV
    (dict(H=0), EINVAL),
    (dict(gate_kind=7), EDTYPE),
    (dict(io_dtype=9), EDTYPE),
    (dict(L=48), EINVAL),                          # not a power of two
    (dict(L=4), EINVAL),                           # L < 2T
    (dict(K=36), EALIGN),                          # K not a multiple of 8
    (dict(V=100), EALIGN),
    (dict(checkpoint=None), EINVAL),
    (dict(rawk=MIS), EALIGN),
    (dict(K=40), EUNSUP),                          # K outside {32, 64, 128}
    (dict(T=17, L=64), EUNSUP),
    (dict(gate_kind=binding.GATE_PER_KEY, L=128), EUNSUP),
    (dict(L=256), EUNSUP),
])
def test_layer_descriptor_errors(lib, kw, want):
    ly = layer(**kw)
    assert verify(lib, ly, cursors()) == want
    assert lib.gdn_spec_verify_path(ctypes.byref(ly)) is None


@pytest.mark.parametrize("kw,path", [
    (dict(), b"tc"),                                        # the Qwen3-Next shape
    (dict(V=256), b"tc"),
    (dict(T=8), b"tc"),
    (dict(T=1), b"tc"),                                     # decode
    (dict(gate_kind=binding.GATE_PER_KEY), b"tc_kda"),     # KDA
    (dict(gate_kind=binding.GATE_PER_KEY, T=8), b"tc_kda"),
    (dict(gate_kind=binding.GATE_PER_KEY, K=64), b"generic"),
    (dict(gate_kind=binding.GATE_PER_KEY, io_dtype=binding.DTYPE_FP32), b"generic"),
    (dict(io_dtype=binding.DTYPE_FP32), b"generic"),
    (dict(L=128), b"generic"),
    (dict(T=9, L=64), b"generic"),
    (dict(K=64), b"generic"),
    (dict(V=96), b"generic"),
])
def test_verify_path_by_shape(lib, kw, path):
    assert lib.gdn_spec_verify_path(ctypes.byref(layer(**kw))) == path


@pytest.mark.parametrize("kw,path", [
    (dict(), b"chunk"),                                     # the Qwen3-Next shape
    (dict(V=256), b"chunk"),
    (dict(L=128), b"chunk"),                                # prefill does not use the ring
    (dict(gate_kind=binding.GATE_PER_KEY), b"sequential"), # KDA
    (dict(io_dtype=binding.DTYPE_FP32), b"sequential"),
    (dict(K=64), b"sequential"),
    (dict(V=96), b"sequential"),
])
def test_prefill_path_by_shape(lib, kw, path):
    lib.gdn_spec_prefill_path.restype = ctypes.c_char_p
    assert lib.gdn_spec_prefill_path(ctypes.byref(layer(**kw))) == path
    assert lib.gdn_spec_prefill_path(ctypes.byref(layer(K=36))) is None


def test_verify_call_errors(lib):
    ly, cu = layer(), cursors()
    assert verify(lib, ly, None) == EINVAL
    assert verify(lib, ly, cursors(num_slots=9)) == EINVAL        # pool sizes differ
    assert verify(lib, ly, cursors(status=None)) == EINVAL
    assert verify(lib, ly, cu, B=-1) == EINVAL
    assert verify(lib, ly, cu, B=0) == OK                          # nothing to do, nothing launched
    assert verify(lib, ly, cu, slot=None) == EINVAL
    assert verify(lib, ly, cu, q=None) == EINVAL
    assert verify(lib, ly, cu, q=MIS) == EALIGN
    assert verify(lib, ly, cu, out=MIS) == EALIGN


def test_commit_reset_and_status_errors(lib):
    cu = cursors()
    commit = lambda T, L, B, slot=FAKE, acc=FAKE: lib.gdn_spec_commit(  # noqa: E731
        ctypes.byref(cu), T, L, slot, B, acc, None)
    assert commit(0, 8, 1) == EINVAL
    assert commit(4, 12, 1) == EINVAL
    assert commit(4, 4, 1) == EINVAL
    assert commit(4, 8, -1) == EINVAL
    assert commit(4, 8, 0) == OK
    assert commit(4, 8, 1, slot=None) == EINVAL
    assert commit(4, 8, 1, acc=None) == EINVAL
    assert lib.gdn_spec_commit(None, 4, 8, FAKE, 1, FAKE, None) == EINVAL
    assert lib.gdn_spec_reset(ctypes.byref(cu), FAKE, -1, None) == EINVAL
    assert lib.gdn_spec_reset(ctypes.byref(cu), FAKE, 0, None) == OK
    assert lib.gdn_spec_reset(ctypes.byref(cu), None, 1, None) == EINVAL
    assert lib.gdn_spec_read_status(ctypes.byref(cu), None, 0, None) == EINVAL
    assert lib.gdn_spec_read_status(None, ctypes.byref(ctypes.c_uint32()), 0, None) == EINVAL


def test_fold_errors(lib):
    cu = cursors()
    two = (binding.LayerDesc * 2)(layer(), layer())
    assert lib.gdn_spec_fold(None, 1, ctypes.byref(cu), FAKE, 1, None) == EINVAL
    assert lib.gdn_spec_fold(two, 0, ctypes.byref(cu), FAKE, 1, None) == EINVAL
    assert lib.gdn_spec_fold(two, 2, ctypes.byref(cu), FAKE, -1, None) == EINVAL
    assert lib.gdn_spec_fold(two, 2, ctypes.byref(cu), FAKE, 0, None) == OK
    assert lib.gdn_spec_fold(two, 2, ctypes.byref(cu), None, 1, None) == EINVAL
    assert lib.gdn_spec_fold(two, 2, ctypes.byref(cursors(num_slots=4)), FAKE, 1, None) == EINVAL
    mixed = (binding.LayerDesc * 2)(layer(), layer(T=2))          # layers must share a shape
    assert lib.gdn_spec_fold(mixed, 2, ctypes.byref(cu), FAKE, 1, None) == EINVAL
    bad = (binding.LayerDesc * 2)(layer(), layer(io_dtype=9))
    assert lib.gdn_spec_fold(bad, 2, ctypes.byref(cu), FAKE, 1, None) == EDTYPE


def test_prefill_and_snapshot_errors(lib):
    ly, cu = layer(), cursors()
    L_, C_ = ctypes.byref(ly), ctypes.byref(cu)
    prefill = lambda B, N, slot=FAKE, q=FAKE, out=FAKE: lib.gdn_spec_prefill(  # noqa: E731
        L_, C_, slot, B, N, q, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, out, 1, None)
    assert prefill(-1, 4) == EINVAL
    assert prefill(1, -4) == EINVAL
    assert prefill(0, 4) == OK
    assert prefill(1, 4, slot=None) == EINVAL
    assert prefill(1, 4, q=None) == EINVAL
    assert prefill(1, 4, out=MIS) == EALIGN
    assert lib.gdn_spec_prefill(ctypes.byref(layer(K=40)), C_, FAKE, 1, 4, *([FAKE] * 8), 1,
                                None) == EUNSUP
    snap_v = lambda B, snap=FAKE, q=FAKE: lib.gdn_spec_snapshot_verify(  # noqa: E731
        L_, C_, FAKE, B, q, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, snap, None)
    assert snap_v(-1) == EINVAL
    assert snap_v(0) == OK
    assert snap_v(1, snap=None) == EINVAL
    assert snap_v(1, snap=MIS) == EALIGN
    assert snap_v(1, q=MIS) == EALIGN
    snap_c = lambda B, acc=FAKE, snap=FAKE: lib.gdn_spec_snapshot_commit(  # noqa: E731
        L_, C_, FAKE, B, acc, snap, None)
    assert snap_c(-1) == EINVAL
    assert snap_c(0) == OK
    assert snap_c(1, acc=None) == EINVAL
    assert snap_c(1, snap=MIS) == EALIGN


def verify_d(lib, ly, cu, B=1, dring=FAKE, slot=FAKE, q=FAKE, out=FAKE):
    return lib.gdn_spec_verify_d(_ref(ly), dring, _ref(cu), slot, B, q, FAKE, FAKE, FAKE, FAKE, FAKE,
                                 FAKE, out, None)


def test_verify_d_errors(lib):
    """The derived-d comparison variant: the tensor-core shapes only, a d ring
    that is present and 16-byte aligned, and the verify call's other checks."""
    ly, cu = layer(), cursors()
    assert verify_d(lib, ly, cu, B=0) == OK
    assert verify_d(lib, ly, cu, dring=None) == EINVAL
    assert verify_d(lib, ly, cu, dring=MIS) == EALIGN
    assert verify_d(lib, ly, None) == EINVAL
    assert verify_d(lib, ly, cu, q=MIS) == EALIGN
    assert verify_d(lib, layer(HV=24), cu) == EINVAL
    for kw in (dict(io_dtype=binding.DTYPE_FP32), dict(gate_kind=binding.GATE_PER_KEY),
               dict(K=64), dict(L=128), dict(T=9, L=64), dict(V=96)):
        assert verify_d(lib, layer(**kw), cu) == EUNSUP, kw
