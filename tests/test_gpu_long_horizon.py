"""Flush-heavy long horizon on the GPU, tracked against the fp64 oracle.

Workload: C1 heads (H=16, HV=32, K=V=128, bf16 I/O) at B=16 with a ring of
L=16, so gdn_spec_fold fires every few commits; accept_len mixes partial and
full accepts (U{1..4}, at least a quarter of rows accept all 4); 16384
committed tokens per slot.  The GPU runs all 16 rows; the oracle follows rows
0 and 1 (all heads) through the same protocol.  Every 512 committed tokens the
outputs of those rows and their folded checkpoints are compared (max-abs
<= 3e-2, relative Frobenius <= 1e-3); the error log is printed.

This is the situation in which the pages' chunked flush drifted on long
outputs (blog post on sglang PR #28695, §12.5-12.7): the exact fold keeps the
checkpoint on the contractive recurrence, so the error must not grow.
"""
import numpy as np
import pytest

import oracle
from gated_delta_rule_spec_gb300 import binding
from gated_delta_rule_spec_gb300 import inputs as gen
from tests.harness import CKPT_REL_FRO, NTHREADS, OUT_TOL_BF16, Scenario, to_dev, to_host

pytestmark = pytest.mark.gpu

TRACKED = (0, 1)


def test_c3_flush_heavy_16k_tokens():
    wl = gen.WORKLOADS["C3"]
    total = wl.extra["committed_tokens"]
    log_every = wl.extra["log_every"]
    sc = Scenario(wl, B=wl.B, seed=3, num_slots=wl.B + 2)
    d = sc.dims
    mask = np.zeros((wl.B, d.HV), np.uint8)
    mask[list(TRACKED)] = 1
    tracked_slots = sc.slot_idx[list(TRACKED)]
    committed = np.zeros(wl.B, np.int64)
    next_log = log_every
    log = []
    folds = 0
    while committed.min() < total:
        w = sc.window()
        dev = {name: to_dev(x) for name, x in w.items()}
        out = binding.verify(sc.layer, sc.cur, sc.slot_dev, dev["q"], dev["k"], dev["v"],
                             dev["a"], dev["b"], sc.A_log_dev, sc.dt_bias_dev)
        f = {name: gen.to_f64(x) for name, x in w.items()}
        o_orc, st = oracle.verify(d, sc.orc, sc.orc_cur, sc.slot_idx, f["q"], f["k"], f["v"],
                                  f["a"], f["b"], sc.A_log, sc.dt_bias, unit_mask=mask,
                                  nthreads=NTHREADS)
        assert st == 0
        acc = gen.accept_lens(sc.rng, wl.B, d.T, full_frac=0.25)
        binding.commit(sc.cur, d.T, d.L, sc.slot_dev, to_dev(acc))
        binding.fold(sc.layer, sc.cur, sc.slot_dev)
        assert oracle.commit(d, sc.orc_cur, tracked_slots, acc[list(TRACKED)]) == 0
        folds += int(sc.orc_cur.is_flush[tracked_slots[0]])
        assert oracle.fold(d, sc.orc, sc.orc_cur, tracked_slots, nthreads=NTHREADS) == 0
        committed += acc
        if committed[TRACKED[0]] >= next_log:
            next_log += log_every
            e_out = sc.out_error(out, o_orc, rows=list(TRACKED))
            e_ck = sc.ckpt_error_per_slot(list(tracked_slots))
            for name in ("write_pos", "cache_base", "is_flush"):
                got = to_host(getattr(sc.cur, name))[tracked_slots]
                assert np.array_equal(got, getattr(sc.orc_cur, name)[tracked_slots]), name
            log.append((int(committed[TRACKED[0]]), e_out, e_ck))
            assert e_out <= OUT_TOL_BF16, log[-1]
            assert e_ck <= CKPT_REL_FRO, log[-1]
    assert binding.read_status(sc.cur) == 0
    assert folds > total // (d.L - d.T)  # the fold really fired every few commits
    print("C3 error log (committed tokens, max-abs output, checkpoint rel-Fro):")
    for row in log:
        print(f"  {row[0]:6d}  {row[1]:.3e}  {row[2]:.3e}")
    # no growth: the last quarter's worst checkpoint error is within 4x the first quarter's
    q = max(1, len(log) // 4)
    first = max(r[2] for r in log[:q])
    last = max(r[2] for r in log[-q:])
    assert last <= 4 * first + 1e-6, (first, last)
