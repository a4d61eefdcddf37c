"""GPU checks of stream order for the kernels launched with programmatic
dependent launch (commit, fold, cursor move).

Such a kernel may start while the kernel before it in the stream is still
running, and must not read anything before its grid-dependency wait.  Here a
torch kernel writes each round's accept lengths into the commit's input
buffer immediately before the commit (a fill, then an add of the new values),
and unrelated torch kernels run between the commit and the fold and between
the fold and the next verify.  A kernel that read its inputs before the wait
would commit stale accept lengths or fold with stale flags; the cursors are
compared with the oracle's bit for bit after every call, the outputs and the
folded checkpoints within the usual bars.
"""
import numpy as np
import pytest
import torch

import oracle
from gated_delta_rule_spec_gb300 import binding
from gated_delta_rule_spec_gb300 import inputs as gen
from tests.harness import CKPT_REL_FRO, NTHREADS, Scenario, to_dev

pytestmark = pytest.mark.gpu


def test_inputs_written_by_the_kernel_just_before():
    wl = gen.WORKLOADS["C2"]
    sc = Scenario(wl, B=8, seed=61, num_slots=24, random_cursors=True)
    assert binding.verify_path(sc.layer) == "tc"
    d = sc.dims
    acc_dev = torch.zeros(sc.B, dtype=torch.int32, device="cuda")
    other = torch.zeros(1 << 20, dtype=torch.float32, device="cuda")
    folds = 0
    for r in range(40):
        w = sc.window()
        out, o_orc, st = sc.verify(w)
        assert st == 0
        assert sc.out_error(out, o_orc) <= sc.out_tol(), f"round {r}"
        acc = gen.accept_lens(sc.rng, sc.B, d.T, full_frac=0.5)
        src = to_dev(acc)
        acc_dev.zero_()          # kernels writing the commit's input right before it
        acc_dev.add_(src)
        binding.commit(sc.cur, d.T, d.L, sc.slot_dev, acc_dev)
        assert oracle.commit(d, sc.orc_cur, sc.slot_idx, acc) == 0
        sc.check_cursors()
        other.add_(1.0)          # an unrelated kernel between commit and fold
        folds += int(sc.orc_cur.is_flush[sc.slot_idx].sum())
        binding.fold(sc.layer, sc.cur, sc.slot_dev)
        assert oracle.fold(d, sc.orc, sc.orc_cur, sc.slot_idx, nthreads=NTHREADS) == 0
        sc.check_cursors()
        other.mul_(0.5)          # and one between the fold and the next verify
    assert binding.read_status(sc.cur) == 0
    assert folds > 0
    used = sorted(set(int(s) for s in sc.slot_idx if s >= 0))
    assert sc.ckpt_error_per_slot(used) <= CKPT_REL_FRO
