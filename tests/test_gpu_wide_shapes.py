"""GPU parity on shapes at the edges of the kernels' ranges, against the oracle.

Tensor-core verify: windows of 6 and 8 tokens (its eight-column template), V = 256
(two units per row and v-head), and a fold deferred until the ring is full (the
second pass of its key phase).  CUDA-core verify: two V-blocks with fp32 I/O, and KDA
with an eight-token window.  This file sorts after the others, so a failure here
leaves the established parity runs complete.
"""
import numpy as np
import pytest

from gated_delta_rule_spec_gb300 import binding
from gated_delta_rule_spec_gb300 import inputs as gen
from tests.harness import CKPT_REL_FRO, Scenario
from tests.test_gpu_kda import _kda_rounds
from tests.test_gpu_parity import _rounds

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("T,L", [(8, 32), (6, 16)])
def test_tc_windows_of_five_to_eight_tokens(T, L):
    """Draft windows of 5..8 tokens on the tensor-core kernel (its eight-column
    template; with T = 6 the query rows 6 and 7 stay zero)."""
    wl = gen.Workload(f"tc-window{T}", B=3, H=2, HV=4, K=128, V=128, T=T, L=L, prefix=16)
    sc = Scenario(wl, B=3, seed=11 + T, num_slots=5, decay_shift=2.0)
    assert binding.verify_path(sc.layer) == "tc"
    _rounds(sc, 20, full_frac=0.3, check_ring_every=2)


def test_tc_two_v_blocks():
    """V = 256: two units per (row, v-head), the v history staged one record per
    copy, raw keys and gates written by V-block 0 only."""
    wl = gen.Workload("tc-v256", B=3, H=2, HV=4, K=128, V=256, T=4, L=16, prefix=16)
    sc = Scenario(wl, B=3, seed=21, num_slots=5, decay_shift=2.0)
    assert binding.verify_path(sc.layer) == "tc"
    _rounds(sc, 20, full_frac=0.3, check_ring_every=2)


def test_tc_fold_deferred_until_the_ring_is_full():
    """The caller may defer the fold while write_pos + T <= L: with T = 8, L = 64
    and full accepts, write_pos climbs 0, 8, .., 56, so the last verify has 64
    keys and its queries in rows 64..71 of the key buffer (the second pass of
    its key phase); the fold then replays a full ring of 64 records."""
    wl = gen.Workload("tc-full-ring", B=2, H=2, HV=4, K=128, V=128, T=8, L=64, prefix=16)
    sc = Scenario(wl, B=2, seed=31, num_slots=4, decay_shift=2.0)
    assert binding.verify_path(sc.layer) == "tc"
    full = np.full(sc.B, wl.T, np.int32)
    for r in range(wl.L // wl.T):
        out, o_orc, st = sc.verify(sc.window())
        assert st == 0
        err = sc.out_error(out, o_orc)
        assert err <= sc.out_tol(), f"write_pos {r * wl.T}: output error {err}"
        sc.check_ring()
        assert sc.commit(full) == 0
        sc.check_cursors()
    assert sc.fold() == 0
    sc.check_cursors()
    assert sc.ckpt_error_per_slot(sorted(set(sc.slot_idx.tolist()))) <= CKPT_REL_FRO
    out, o_orc, st = sc.verify(sc.window())
    assert st == 0 and sc.out_error(out, o_orc) <= sc.out_tol()
    assert binding.read_status(sc.cur) == 0


def test_generic_two_v_blocks_fp32():
    """The CUDA-core kernel over V = 160: a full and a partial block of 128 state
    rows (and fold items of 64, 64 and 32 rows)."""
    wl = gen.Workload("generic-v160", B=2, H=1, HV=2, K=64, V=160, T=3, L=16, io_dtype=gen.FP32,
                      prefix=8)
    sc = Scenario(wl, B=2, seed=41, num_slots=3)
    assert binding.verify_path(sc.layer) == "generic"
    worst = _rounds(sc, 12, full_frac=0.3)
    assert worst["out"] <= 1e-4


def test_kda_window_of_eight_tokens():
    """KDA with a draft window of eight tokens and K = V = 64, bf16."""
    wl = gen.Workload("kda-t8", B=2, H=2, HV=4, K=64, V=64, T=8, L=32, per_key_gate=True,
                      prefix=16)
    sc = Scenario(wl, B=2, seed=13, num_slots=3, decay_shift=2.0)
    assert binding.verify_path(sc.layer) == "generic"
    _kda_rounds(sc, 15, ring_every=3)


@pytest.mark.parametrize("H,HV", [(4, 4), (2, 6)])
def test_tc_single_head_units_odd_groups(H, HV):
    """An odd number of v-heads per q/k head (G = 1, G = 3): the tensor-core
    kernel takes one v-head per unit instead of a pair."""
    wl = gen.Workload(f"tc-g{HV // H}", B=3, H=H, HV=HV, K=128, V=128, T=4, L=16, prefix=16)
    sc = Scenario(wl, B=3, seed=51 + HV, num_slots=5, decay_shift=2.0, random_cursors=True)
    assert binding.verify_path(sc.layer) == "tc"
    _rounds(sc, 16, full_frac=0.3, check_ring_every=2)
