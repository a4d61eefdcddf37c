"""GPU parity of the tensor-core KDA verify ("tc_kda") against the oracle.

The per-key gate puts the decay inside the contraction over K; the kernel
factors it through 16-token block boundaries, takes the blocks below the
diagonal from one tf32 MMA per target block and the diagonal blocks from
running products on the CUDA cores.  These cases stress each piece: windows
of 1, 4 and 8 tokens (queries in the last block or across a block boundary),
ring fills that end inside and on block boundaries, two blocks of 128 state
rows, v-heads sharing a q/k head, raw (non-unit) keys and queries, decays from
almost none to underflowing within a block, and a checkpoint-tile wait that
runs out.
"""
import numpy as np
import pytest

from gated_delta_rule_spec_gb300 import binding
from gated_delta_rule_spec_gb300 import inputs as gen
from tests.harness import Scenario, to_dev
from tests.test_gpu_kda import _kda_rounds

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("T,L", [(1, 64), (4, 64), (8, 64), (4, 32)])
def test_tc_kda_windows(T, L):
    wl = gen.Workload(f"kda-tc-t{T}-l{L}", B=3, H=2, HV=4, K=128, V=128, T=T, L=L, per_key_gate=True,
                      prefix=16)
    sc = Scenario(wl, B=3, seed=70 + T + L, num_slots=5, random_cursors=True)
    assert binding.verify_path(sc.layer) == "tc_kda"
    worst = _kda_rounds(sc, 40, ring_every=4)
    print(f"tc_kda T={T} L={L}: max-abs output error {worst:.3e}")


@pytest.mark.parametrize("shift", [-4.0, 0.0, 6.0])
def test_tc_kda_decay_regimes(shift):
    """shift -4: per-channel decays that underflow inside a block; +6: almost
    no decay, so every block's products stay near one."""
    wl = gen.Workload("kda-tc-decay", B=2, H=2, HV=4, K=128, V=128, T=4, L=64, per_key_gate=True,
                      prefix=16)
    sc = Scenario(wl, B=2, seed=90, num_slots=3, decay_shift=shift, random_cursors=True)
    assert binding.verify_path(sc.layer) == "tc_kda"
    worst = _kda_rounds(sc, 60, ring_every=6)
    print(f"tc_kda decay shift {shift}: max-abs output error {worst:.3e}")


def test_tc_kda_wide_v_raw_keys():
    """V = 256 (two blocks of state rows), G = 2, raw q/k scaled over [0.25, 4]."""
    wl = gen.Workload("kda-tc-v256", B=2, H=2, HV=4, K=128, V=256, T=4, L=64, per_key_gate=True,
                      prefix=16)
    sc = Scenario(wl, B=2, seed=95, num_slots=4, key_scale=(0.25, 4.0), random_cursors=True)
    assert binding.verify_path(sc.layer) == "tc_kda"
    worst = _kda_rounds(sc, 30, ring_every=3)
    print(f"tc_kda V=256 raw keys: max-abs output error {worst:.3e}")


def test_tc_kda_tile_wait_runs_out_then_recovers():
    wl = gen.Workload("kda-tc-timeout", B=3, H=2, HV=4, K=128, V=128, T=4, L=32, per_key_gate=True,
                      prefix=16)
    sc = Scenario(wl, B=3, seed=97, num_slots=5, random_cursors=True)
    assert binding.verify_path(sc.layer) == "tc_kda"
    w = sc.window()
    dev = {n: to_dev(x) for n, x in w.items()}
    prev = binding.set_wait_limit(0)
    try:
        binding.verify(sc.layer, sc.cur, sc.slot_dev, dev["q"], dev["k"], dev["v"], dev["a"], dev["b"],
                       sc.A_log_dev, sc.dt_bias_dev)
        st = binding.read_status(sc.cur)
    finally:
        binding.set_wait_limit(binding.WAIT_LIMIT_DEFAULT)
    assert prev == 1 << 20
    assert st & binding.ST_TIMEOUT
    out, o_orc, st2 = sc.verify(w)
    assert st2 == 0 and binding.read_status(sc.cur) == 0
    assert sc.out_error(out, o_orc) <= sc.out_tol()
    sc.check_ring()
    sc.check_cursors()
