"""Plain decode (a window of one token) through the same calls, checkpoint,
ring and cursors as spec-verify, against the oracle.

The pages' decode and verify share one set of data structures (checkpoint +
ring + three cursors) and differ only in the window length: 1 for decode, the
draft window for verify (blog post on sglang PR #28695, §12.9).  Every round
verifies one token per row, commits it (accept_len = 1, as in decode) and
folds the rows whose ring is full.
"""
import pytest

from gated_delta_rule_spec_gb300 import binding
from gated_delta_rule_spec_gb300 import inputs as gen
from tests.harness import CKPT_REL_FRO, Scenario

pytestmark = pytest.mark.gpu


def _decode_rounds(sc, rounds, ring_every):
    worst = 0.0
    folds = 0
    for r in range(rounds):
        w = sc.window()
        out, o_orc, st = sc.verify(w)
        assert st == 0
        err = sc.out_error(out, o_orc)
        worst = max(worst, err)
        assert err <= sc.out_tol(), f"round {r}: output error {err}"
        if r % ring_every == 0:
            sc.check_ring()
        acc = gen.accept_lens(sc.rng, sc.B, 1)
        assert (acc == 1).all()
        assert sc.commit(acc) == 0
        folds += int(sc.orc_cur.is_flush[sc.slot_idx].sum())
        assert sc.fold() == 0
        sc.check_cursors()
        assert sc.ckpt_error_per_slot(sorted(set(sc.slot_idx.tolist()))) <= CKPT_REL_FRO
    assert binding.read_status(sc.cur) == 0
    return worst, folds


def test_decode_qwen3next_shape_tensor_core_path():
    """T = 1 at the Qwen3-Next head shape, L = 64: the ring fills over 63
    decode steps, then folds; scattered slots with random starting cursors."""
    wl = gen.Workload("qwen3next-decode", B=8, H=16, HV=32, K=128, V=128, T=1, L=64, prefix=16)
    sc = Scenario(wl, B=8, seed=21, num_slots=24, random_cursors=True)
    assert binding.verify_path(sc.layer) == "tc"
    worst, folds = _decode_rounds(sc, 90, ring_every=10)
    assert folds >= 8   # every row's ring filled and folded at least once
    print(f"decode T=1 (tc): max-abs output error {worst:.3e}, {folds} row folds")


def test_decode_fp32_generic_path():
    """T = 1 on the CUDA-core path with fp32 I/O: the error is a number, near
    fp32 rounding."""
    wl = gen.Workload("decode-tiny-fp32", B=2, H=2, HV=4, K=32, V=32, T=1, L=8, io_dtype=gen.FP32,
                      prefix=6)
    sc = Scenario(wl, B=2, seed=22, num_slots=3)
    assert binding.verify_path(sc.layer) == "generic"
    worst, folds = _decode_rounds(sc, 30, ring_every=1)
    assert folds >= 2
    assert worst <= 1e-4
    print(f"decode T=1 (generic, fp32): max-abs output error {worst:.3e}")
