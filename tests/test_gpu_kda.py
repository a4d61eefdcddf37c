"""GPU parity of the KDA variant (one gate per key channel) against the oracle.

Workload: H=16, HV=32, K=V=128, bf16 I/O, fp32 checkpoint, T=4, L=64, at B=1
and B=64, 200 verify -> commit -> fold rounds with accept_len ~ U{1..4}.
"""
import pytest

from gated_delta_rule_spec_gb300 import binding
from gated_delta_rule_spec_gb300 import inputs as gen
from tests.harness import CKPT_REL_FRO, Scenario

pytestmark = pytest.mark.gpu


def _kda_rounds(sc, rounds, ring_every):
    worst = 0.0
    for r in range(rounds):
        w = sc.window()
        out, o_orc, st = sc.verify(w)
        assert st == 0
        err = sc.out_error(out, o_orc)
        worst = max(worst, err)
        assert err <= sc.out_tol(), f"round {r}: {err}"
        if r % ring_every == 0:
            sc.check_ring()
        acc = gen.accept_lens(sc.rng, sc.B, sc.dims.T)
        assert sc.commit(acc) == 0
        assert sc.fold() == 0
        sc.check_cursors()
        assert sc.ckpt_error_per_slot(sorted(set(sc.slot_idx.tolist()))) <= CKPT_REL_FRO
    assert binding.read_status(sc.cur) == 0
    return worst


@pytest.mark.parametrize("B,rounds", [(1, 200), (64, 200)])
def test_c4_kda_rounds(B, rounds):
    wl = gen.WORKLOADS["C4"]
    sc = Scenario(wl, B=B, seed=4, num_slots=B + 3)
    worst = _kda_rounds(sc, rounds, ring_every=20 if B > 1 else 5)
    print(f"C4 KDA B={B}: max-abs output error {worst:.3e}")


def test_kda_small_weak_decay_fp32():
    wl = gen.Workload("kda-tiny", B=2, H=2, HV=4, K=32, V=16, T=3, L=16, io_dtype=gen.FP32,
                      per_key_gate=True, prefix=12)
    sc = Scenario(wl, B=2, seed=9, num_slots=4, decay_shift=4.0)
    worst = _kda_rounds(sc, 25, ring_every=1)
    assert worst <= 1e-4

