"""GPU parity of the chunk-parallel prefill (tensor cores) against the oracle.

gdn_spec_prefill takes the chunk-parallel path for the scalar gate with bf16
I/O, K = 128 and V a multiple of 128: the chunked UT form that the blog post
on sglang PR #28695 (appendix B.1) names as the prefill authority, 64 tokens
per step, with the state carried in tensor memory.  These cases span many
chunks and ragged tails, two 128-row blocks of V, grouped heads, raw
(non-unit) keys and queries, decays from nearly none to underflowing, a
continuation from the checkpoint, the empty prompt, and a wait that runs out.
The bars are the path's stated tolerances: outputs within 3e-2 max-abs (bf16),
the checkpoint within 1e-3 relative Frobenius.
"""
import numpy as np
import pytest
import torch

import oracle
from gated_delta_rule_spec_gb300 import binding
from gated_delta_rule_spec_gb300 import inputs as gen
from tests.harness import CKPT_REL_FRO, NTHREADS, OUT_TOL_BF16, to_dev, to_host
from tests.test_gpu_prefill import PrefillCase

pytestmark = pytest.mark.gpu


def _run(c, slots, w, from_zero):
    f = {n: gen.to_f64(x) for n, x in w.items()}
    o_orc, st_orc = oracle.prefill(c.d, c.orc, c.orc_cur, slots, f["q"], f["k"], f["v"], f["a"], f["b"],
                                   c.A_log.astype(np.float64), c.dt_bias.astype(np.float64),
                                   from_zero=from_zero, nthreads=NTHREADS)
    dev = {n: to_dev(x) for n, x in w.items()}
    out = binding.prefill(c.layer, c.cur, to_dev(slots), dev["q"], dev["k"], dev["v"], dev["a"], dev["b"],
                          torch.from_numpy(c.A_log).cuda(), torch.from_numpy(c.dt_bias).cuda(),
                          from_zero=from_zero)
    st = binding.read_status(c.cur)
    return gen.to_f64(to_host(out)), o_orc, st, st_orc


def _prompt(c, B, N, key_scale=None):
    d = c.d
    return gen.window_inputs(c.rng, B, N, d.H, d.HV, d.K, d.V, gen.BF16, key_scale=key_scale)


@pytest.mark.parametrize("decay", ["layer", "none", "strong"])
def test_chunk_prefill_long_prompt_then_continue(decay):
    """700 tokens from zero (ten full chunks and a ragged one), then 130 more
    from the checkpoints; V = 256 (two state-row blocks), two v-heads per q/k
    head, raw q/k scaled over [0.2, 5]."""
    c = PrefillCase(H=2, HV=4, K=128, V=256, L=64, num_slots=5, io=gen.BF16, per_key=False,
                    seed=201 + ["layer", "none", "strong"].index(decay))
    assert binding.prefill_path(c.layer) == "chunk"
    if decay == "none":        # g close to 0: the state keeps everything it was given
        c.A_log[:] = -8.0
    elif decay == "strong":    # g around -50 per token: the chunk's decays underflow
        c.A_log[:] = np.log(16.0)
        c.dt_bias[:] = 3.0
    slots = np.array([4, -1, 1], np.int32)
    errs = []
    for N, from_zero in ((700, True), (130, False)):
        out, o_orc, st, st_orc = _run(c, slots, _prompt(c, 3, N, key_scale=(0.2, 5.0)), from_zero)
        assert st == st_orc == 0
        err = float(np.max(np.abs(out - o_orc)))
        assert err <= OUT_TOL_BF16, err
        assert not out[1].any()          # padding row reads out zeros
        ck = c.check_state(slots)
        errs.append((err, ck))
    print(f"chunk prefill decay={decay}: " +
          ", ".join(f"max-abs out {e:.2e} / ckpt rel-Fro {k:.2e}" for e, k in errs))


@pytest.mark.parametrize("N", [1, 5, 63, 64, 65, 128])
def test_chunk_prefill_chunk_edges(N):
    """Prompts at and around the 64-token chunk boundary, Qwen3-Next heads."""
    c = PrefillCase(H=16, HV=32, K=128, V=128, L=64, num_slots=3, io=gen.BF16, per_key=False,
                    seed=300 + N)
    slots = np.array([2, 0], np.int32)
    out, o_orc, st, st_orc = _run(c, slots, _prompt(c, 2, N), True)
    assert st == st_orc == 0
    err = float(np.max(np.abs(out - o_orc)))
    assert err <= OUT_TOL_BF16, err
    c.check_state(slots)


def test_chunk_prefill_empty_prompt():
    """N = 0 from zero: the slots' checkpoints become zero and the cursors reset;
    the other slots are bitwise untouched."""
    c = PrefillCase(H=2, HV=4, K=128, V=128, L=64, num_slots=4, io=gen.BF16, per_key=False, seed=311)
    slots = np.array([3, 1], np.int32)
    ck0 = c.layer.checkpoint.clone()
    z = {n: np.zeros((2, 0) + x.shape[2:], x.dtype) for n, x in _prompt(c, 2, 1).items()}
    out, o_orc, st, st_orc = _run(c, slots, z, True)
    assert st == st_orc == 0 and out.size == 0
    ck = to_host(c.layer.checkpoint)
    assert not ck[[1, 3]].any()
    assert torch.equal(c.layer.checkpoint[[0, 2]].view(torch.int32), ck0[[0, 2]].view(torch.int32))
    c.check_state(slots)


def test_chunk_prefill_leaves_other_slots_untouched():
    """Slots outside the batch keep their checkpoints bit for bit."""
    c = PrefillCase(H=2, HV=4, K=128, V=128, L=64, num_slots=6, io=gen.BF16, per_key=False, seed=321)
    slots = np.array([5, 2], np.int32)
    ck0 = c.layer.checkpoint.clone()
    out, o_orc, st, _ = _run(c, slots, _prompt(c, 2, 150), True)
    assert st == 0 and float(np.max(np.abs(out - o_orc))) <= OUT_TOL_BF16
    others = [0, 1, 3, 4]
    assert torch.equal(c.layer.checkpoint[others].view(torch.int32), ck0[others].view(torch.int32))
    c.check_state(slots)


def test_chunk_prefill_wait_runs_out_poisons_rows():
    """A wait on a prompt chunk that gives up at once: TIMEOUT, every computed
    row poisoned (write_pos = -1), slots outside the batch untouched; reset and
    a prefill with the default limit make the rows usable again."""
    c = PrefillCase(H=2, HV=4, K=128, V=128, L=64, num_slots=5, io=gen.BF16, per_key=False, seed=331)
    slots = np.array([4, 0, -1], np.int32)
    ck0 = c.layer.checkpoint.clone()
    wp0 = to_host(c.cur.write_pos).copy()
    w = _prompt(c, 3, 100)
    dev = {n: to_dev(x) for n, x in w.items()}
    prev = binding.set_wait_limit(0)
    try:
        binding.prefill(c.layer, c.cur, to_dev(slots), dev["q"], dev["k"], dev["v"], dev["a"], dev["b"],
                        torch.from_numpy(c.A_log).cuda(), torch.from_numpy(c.dt_bias).cuda(), from_zero=True)
        st = binding.read_status(c.cur)
    finally:
        binding.set_wait_limit(binding.WAIT_LIMIT_DEFAULT)
    assert prev == 1 << 20
    assert st & binding.ST_TIMEOUT
    wp = to_host(c.cur.write_pos)
    for s in range(c.d.num_slots):
        if s in (4, 0):
            assert wp[s] == -1, s
        else:
            assert wp[s] == wp0[s], s
    others = [1, 2, 3]
    assert torch.equal(c.layer.checkpoint[others].view(torch.int32), ck0[others].view(torch.int32))
    # rebuilt: reset, then the same prefill with the default limit matches the oracle
    binding.reset(c.cur, to_dev(slots))
    oracle.reset(c.d, c.orc_cur, slots)
    out, o_orc, st, st_orc = _run(c, slots, w, True)
    assert st == st_orc == 0
    assert float(np.max(np.abs(out - o_orc))) <= OUT_TOL_BF16
    c.check_state(slots)


def test_chunk_prefill_4096_tokens_without_decay():
    """64 chunks with g close to 0: the state keeps everything; the tf32 error of
    the state products does not grow with the prompt (the delta rule corrects
    its own error), measured at about 3e-4 relative Frobenius."""
    c = PrefillCase(H=2, HV=4, K=128, V=128, L=64, num_slots=3, io=gen.BF16, per_key=False, seed=4096)
    c.A_log[:] = -8.0
    slots = np.array([2, 0], np.int32)
    out, o_orc, st, st_orc = _run(c, slots, _prompt(c, 2, 4096), True)
    assert st == st_orc == 0
    err = float(np.max(np.abs(out - o_orc)))
    assert err <= OUT_TOL_BF16, err
    ck = c.check_state(slots)
    print(f"chunk prefill 4096 tokens, no decay: max-abs out {err:.2e}, ckpt rel-Fro {ck:.2e}")


def test_chunk_prefill_bench_size_sampled_rows():
    """The launch the bench times, B = 128 prompts of 256 tokens over a 512-slot
    pool (Qwen3-Next heads, from zero): every row runs on the GPU, and four
    sampled rows are checked against the oracle (rows are independent, so the
    oracle runs on those rows alone)."""
    H, HV, K, V, L, S = 16, 32, 128, 128, 64, 512
    B, N = 128, 256
    rng = gen.rng_for(7, "prefill-bench-size")
    d = oracle.Dims(H=H, HV=HV, K=K, V=V, T=4, L=L, num_slots=S, per_key_gate=False, scale=0.9)
    layer = binding.SpecLayer(H, HV, K, V, 4, L, S, io_dtype="bf16", scale=0.9)
    cur = binding.SpecCursors(S)
    A_log, dt_bias = gen.layer_params(rng, HV, K, False)
    slots = gen.scattered_slots(rng, S, B)
    w = gen.window_inputs(rng, B, N, H, HV, K, V, gen.BF16)
    dev = {n: to_dev(x) for n, x in w.items()}
    out = binding.prefill(layer, cur, to_dev(slots), dev["q"], dev["k"], dev["v"], dev["a"], dev["b"],
                          torch.from_numpy(A_log).cuda(), torch.from_numpy(dt_bias).cuda(), from_zero=True)
    assert binding.read_status(cur) == 0
    got_out = gen.to_f64(to_host(out))
    got_ck = to_host(layer.checkpoint).astype(np.float64)
    sample = np.array([0, 37, 101, 127])
    orc = oracle.Layer(d)
    orc_cur = oracle.Cursors(S, np.zeros(S, np.int32), np.zeros(S, np.int32), np.zeros(S, np.int32))
    f = {n: gen.to_f64(x)[sample] for n, x in w.items()}
    o_orc, st = oracle.prefill(d, orc, orc_cur, slots[sample], f["q"], f["k"], f["v"], f["a"], f["b"],
                               A_log.astype(np.float64), dt_bias.astype(np.float64), from_zero=True,
                               nthreads=NTHREADS)
    assert st == 0
    err = float(np.max(np.abs(got_out[sample] - o_orc)))
    assert err <= OUT_TOL_BF16, err
    worst = 0.0
    for s in slots[sample]:
        ref = orc.checkpoint[s]
        worst = max(worst, np.linalg.norm(got_ck[s] - ref) / np.linalg.norm(ref))
    assert worst <= CKPT_REL_FRO, worst
    wp = to_host(cur.write_pos)
    assert not wp[slots].any()
    print(f"chunk prefill B=128 N=256, 4 sampled rows: max-abs out {err:.2e}, ckpt rel-Fro {worst:.2e}")
