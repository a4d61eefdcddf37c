"""GPU parity of prefill against the oracle.

Prefill runs each row's prompt through the recurrence, writes every token's
output, stores the final state as the slot's checkpoint and resets the slot's
cursors (the prefill -> decode handoff of the blog post on sglang PR #28695,
appendix A.2).  The prompts here span several 64-token chunks and a ragged
tail; the second call of a test continues from the checkpoints (chunked
prefill); decode then runs on the state prefill left.
"""
import numpy as np
import pytest
import torch

import oracle
from gated_delta_rule_spec_gb300 import binding
from gated_delta_rule_spec_gb300 import inputs as gen
from tests.harness import CKPT_REL_FRO, NTHREADS, OUT_TOL_BF16, OUT_TOL_FP32, to_dev, to_host

pytestmark = pytest.mark.gpu


class PrefillCase:
    """A layer with random checkpoints and cursors on both sides."""

    def __init__(self, H, HV, K, V, L, num_slots, io, per_key, seed, T=4):
        self.rng = np.random.default_rng(seed)
        self.io, self.per_key = io, per_key
        self.d = oracle.Dims(H=H, HV=HV, K=K, V=V, T=T, L=L, num_slots=num_slots,
                             per_key_gate=per_key, scale=0.9)
        ck = (self.rng.standard_normal((num_slots, HV, V, K)) * 0.3).astype(np.float32)
        ring = gen.garbage_ring(self.rng, num_slots, H, HV, L, K, V, io, per_key)
        self.orc = oracle.Layer(self.d, checkpoint=ck.astype(np.float64), rawv=gen.to_f64(ring["rawv"]),
                                rawk=gen.to_f64(ring["rawk"]), ring_g=ring["g"].astype(np.float64),
                                ring_beta=ring["beta"].astype(np.float64))
        self.layer = binding.SpecLayer(H, HV, K, V, T, L, num_slots, per_key_gate=per_key,
                                       io_dtype="bf16" if io == gen.BF16 else "fp32", scale=0.9)
        self.layer.checkpoint.copy_(torch.from_numpy(ck))
        wp = self.rng.integers(0, L - 2 * T + 1, num_slots).astype(np.int32)
        base = self.rng.integers(0, L, num_slots).astype(np.int32)
        flag = np.zeros(num_slots, np.int32)
        self.orc_cur = oracle.Cursors(num_slots, wp, base, flag)
        self.cur = binding.SpecCursors(num_slots)
        for n, x in (("write_pos", wp), ("cache_base", base), ("is_flush", flag)):
            getattr(self.cur, n).copy_(torch.from_numpy(x))
        self.A_log, self.dt_bias = gen.layer_params(self.rng, HV, K, per_key)

    def prompt(self, B, N):
        d = self.d
        return gen.window_inputs(self.rng, B, N, d.H, d.HV, d.K, d.V, self.io, self.per_key)

    def prefill(self, slots, w, from_zero):
        f = {n: gen.to_f64(x) for n, x in w.items()}
        o_orc, st_orc = oracle.prefill(self.d, self.orc, self.orc_cur, slots, f["q"], f["k"], f["v"],
                                       f["a"], f["b"], self.A_log.astype(np.float64),
                                       self.dt_bias.astype(np.float64), from_zero=from_zero,
                                       nthreads=NTHREADS)
        dev = {n: to_dev(x) for n, x in w.items()}
        out = binding.prefill(self.layer, self.cur, to_dev(slots), dev["q"], dev["k"], dev["v"],
                              dev["a"], dev["b"], torch.from_numpy(self.A_log).cuda(),
                              torch.from_numpy(self.dt_bias).cuda(), from_zero=from_zero)
        st = binding.read_status(self.cur)
        return gen.to_f64(to_host(out)), o_orc, st, st_orc

    def check_state(self, slots):
        for n in ("write_pos", "cache_base", "is_flush"):
            assert np.array_equal(to_host(getattr(self.cur, n)), getattr(self.orc_cur, n)), n
        got = to_host(self.layer.checkpoint).astype(np.float64)
        worst = 0.0
        for s in range(self.d.num_slots):
            ref = self.orc.checkpoint[s]
            e = np.linalg.norm(got[s] - ref) / max(np.linalg.norm(ref), 1e-30)
            worst = max(worst, e)
        assert worst <= CKPT_REL_FRO, worst
        return worst


def _tol(io):
    return OUT_TOL_BF16 if io == gen.BF16 else OUT_TOL_FP32


@pytest.mark.parametrize("per_key", [False, True])
def test_prefill_qwen3next_shape_then_continue(per_key):
    """Qwen3-Next heads, bf16: 150 prompt tokens from zero (two full chunks and a
    ragged one), then 70 more from the checkpoints; padding and a repeated
    interleaving of slots."""
    c = PrefillCase(H=16, HV=32, K=128, V=128, L=64, num_slots=6, io=gen.BF16, per_key=per_key,
                    seed=61 + per_key)
    assert binding.prefill_path(c.layer) == ("sequential" if per_key else "chunk")
    slots = np.array([5, 1, -1, 3], np.int32)
    out, o_orc, st, st_orc = c.prefill(slots, c.prompt(4, 150), from_zero=True)
    assert st == st_orc == 0
    err = float(np.max(np.abs(out - o_orc)))
    assert err <= _tol(c.io), err
    assert not out[2].any()                 # padding row reads out zeros
    c.check_state(slots)
    out, o_orc, st, st_orc = c.prefill(slots, c.prompt(4, 70), from_zero=False)
    assert st == st_orc == 0
    err2 = float(np.max(np.abs(out - o_orc)))
    assert err2 <= _tol(c.io), err2
    ck = c.check_state(slots)
    print(f"prefill per_key={per_key}: max-abs output error {err:.3e} / {err2:.3e}, "
          f"checkpoint rel-Frobenius {ck:.2e}")


def test_prefill_fp32_small_heads_error_is_a_number():
    c = PrefillCase(H=2, HV=4, K=32, V=40, L=16, num_slots=3, io=gen.FP32, per_key=False, seed=71)
    assert binding.prefill_path(c.layer) == "sequential"
    slots = np.array([2, 0], np.int32)
    out, o_orc, st, _ = c.prefill(slots, c.prompt(2, 97), from_zero=True)
    assert st == 0
    err = float(np.max(np.abs(out - o_orc)))
    assert err <= 1e-4
    c.check_state(slots)
    print(f"prefill fp32 (V = 40: one partial 64-row block): max-abs output error {err:.3e}")


def test_prefill_status_rules():
    """Out-of-range slot, and a slot with unfolded records when continuing:
    both skipped (zeros out, state and cursors untouched), status bits set."""
    c = PrefillCase(H=2, HV=2, K=64, V=64, L=16, num_slots=4, io=gen.BF16, per_key=False, seed=81)
    c.orc_cur.write_pos[:] = [0, 3, 0, 0]
    c.cur.write_pos.copy_(torch.from_numpy(c.orc_cur.write_pos))
    slots = np.array([9, 1, 2], np.int32)
    ck1 = to_host(c.layer.checkpoint)[1].copy()
    out, o_orc, st, st_orc = c.prefill(slots, c.prompt(3, 5), from_zero=False)
    assert st == st_orc == binding.ST_SLOT_OOR | binding.ST_UNFOLDED
    assert not out[:2].any() and out[2].any()
    assert np.array_equal(to_host(c.layer.checkpoint)[1], ck1)
    c.check_state(slots)


def test_prefill_then_decode_matches_oracle():
    """The handoff: after prefill, verify -> commit -> fold rounds run on the
    prefilled checkpoint and the reset cursors."""
    c = PrefillCase(H=16, HV=32, K=128, V=128, L=64, num_slots=3, io=gen.BF16, per_key=False,
                    seed=91)
    slots = np.array([2, 0], np.int32)
    c.prefill(slots, c.prompt(2, 40), from_zero=True)
    d = c.d
    for r in range(20):
        w = gen.window_inputs(c.rng, 2, d.T, d.H, d.HV, d.K, d.V, gen.BF16)
        f = {n: gen.to_f64(x) for n, x in w.items()}
        o_orc, _ = oracle.verify(d, c.orc, c.orc_cur, slots, f["q"], f["k"], f["v"], f["a"], f["b"],
                                 c.A_log.astype(np.float64), c.dt_bias.astype(np.float64),
                                 nthreads=NTHREADS)
        dev = {n: to_dev(x) for n, x in w.items()}
        out = binding.verify(c.layer, c.cur, to_dev(slots), dev["q"], dev["k"], dev["v"], dev["a"],
                             dev["b"], torch.from_numpy(c.A_log).cuda(),
                             torch.from_numpy(c.dt_bias).cuda())
        err = float(np.max(np.abs(gen.to_f64(to_host(out)) - o_orc)))
        assert err <= OUT_TOL_BF16, f"round {r}: {err}"
        acc = gen.accept_lens(c.rng, 2, d.T)
        assert oracle.commit(d, c.orc_cur, slots, acc) == 0
        binding.commit(c.cur, d.T, d.L, to_dev(slots), to_dev(acc))
        oracle.fold(d, c.orc, c.orc_cur, slots, nthreads=NTHREADS)
        binding.fold(c.layer, c.cur, to_dev(slots))
        c.check_state(slots)
    assert binding.read_status(c.cur) == 0
