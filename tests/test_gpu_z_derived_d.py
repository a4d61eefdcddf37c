"""GPU parity of the derived-d comparison variant (gdn_spec_verify_d) against
the oracle's verify_d: a ring that also caches every token's corrected delta
d_t = beta_t (v_t - S_t^- k^_t), the first design of the blog post on sglang PR
#28695 (§12.1, appendix A.1).  With a window of one token it is the no-inverse
decode of that design (§12.2, §12.9, Part A).

Each run starts from a prefilled checkpoint with an empty ring, so every
history record's d in the d ring was written by an earlier verify_d of the
same run; commit and fold are the ring path's (the fold replays raw records).
Bars: outputs and the window's d within 3e-2 max-abs (bf16 I/O), ring records
and cursors bit-exact, each folded (slot, v-head) checkpoint within 1e-3
relative Frobenius error.
"""
import numpy as np
import pytest

from gated_delta_rule_spec_gb300 import binding
from gated_delta_rule_spec_gb300 import inputs as gen
from tests.harness import CKPT_REL_FRO, OUT_TOL_BF16, Scenario

pytestmark = pytest.mark.gpu

D_TOL = 3e-2


def _d_rounds(sc: Scenario, rounds: int, full_frac: float = 0.0):
    dring = sc.layer.new_dring()
    worst = {"out": 0.0, "d": 0.0, "ckpt": 0.0}
    folds = 0
    for r in range(rounds):
        out, o_orc, d_dev, d_orc, st = sc.verify_d(sc.window(), dring)
        assert st == 0
        e_out = sc.out_error(out, o_orc)
        rows = [i for i, s in enumerate(sc.slot_idx) if s >= 0]
        e_d = float(np.max(np.abs(d_dev[rows] - d_orc[rows]))) if rows else 0.0
        worst["out"] = max(worst["out"], e_out)
        worst["d"] = max(worst["d"], e_d)
        assert e_out <= OUT_TOL_BF16, f"round {r}: output error {e_out}"
        assert e_d <= D_TOL, f"round {r}: window d error {e_d}"
        sc.check_ring()
        acc = gen.accept_lens(sc.rng, sc.B, sc.dims.T, full_frac)
        assert sc.commit(acc) == 0
        folds += int(sc.orc_cur.is_flush[[s for s in sc.slot_idx if s >= 0]].sum())
        assert sc.fold() == 0
        sc.check_cursors()
        e = sc.ckpt_error_per_slot(sorted(set(int(s) for s in sc.slot_idx if s >= 0)))
        worst["ckpt"] = max(worst["ckpt"], e)
        assert e <= CKPT_REL_FRO, f"round {r}: checkpoint error {e}"
    assert folds > 0
    assert binding.read_status(sc.cur) == 0
    return worst


def test_derived_d_qwen3next_rounds_with_folds():
    """Qwen3-Next shape, B = 4 (one padding row), 50 rounds: the ring fills to
    the fold margin and folds, so the history d's span several folds."""
    wl = gen.WORKLOADS["C1"]
    sc = Scenario(wl, B=4, seed=121, num_slots=8, slot_idx=np.array([5, -1, 2, 7], np.int32))
    worst = _d_rounds(sc, 50, full_frac=0.3)
    print(f"derived-d: out {worst['out']:.2e}, d {worst['d']:.2e}, ckpt {worst['ckpt']:.2e}")


def test_derived_d_decode_window_of_one():
    """Plain decode (T = 1): the window system is a single token, no inverse."""
    wl = gen.Workload("d-decode", B=6, H=16, HV=32, K=128, V=128, T=1, L=16, prefix=24)
    sc = Scenario(wl, B=6, seed=131, num_slots=9, decay_shift=1.0)
    _d_rounds(sc, 40)


def test_derived_d_window_of_eight_and_two_v_blocks():
    """T = 8 (the eight-column template) with V = 256 (two units per row and v-head)."""
    wl = gen.Workload("d-t8-v256", B=2, H=2, HV=4, K=128, V=256, T=8, L=32, prefix=16)
    sc = Scenario(wl, B=2, seed=141, num_slots=3, decay_shift=2.0)
    _d_rounds(sc, 24, full_frac=0.3)
