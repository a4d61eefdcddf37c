"""The bounded-wait path on the GPU, made to run out on purpose and safely.

gdn_spec_set_wait_limit(0) makes the first wait on each asynchronous data copy
give up at once (the tensor-core verify's checkpoint tile, the fold's ring
records).  The copy itself is still drained with the normal limit before its
buffer is reused, so nothing stays in flight: the call reports
GDN_SPEC_ST_TIMEOUT and returns.  Afterwards, with the default limit back:

* verify: the same window on the same buffers matches the oracle again (its
  outputs, and the ring, whose window records the failed call may have written
  only in part);
* fold: every row it was asked to fold is poisoned (write_pos = -1), the other
  rows and every checkpoint it did not touch are bitwise as before, later
  calls report CURSOR_CORRUPT for the poisoned rows, and gdn_spec_reset plus a
  prefill make them usable again.
"""
import numpy as np
import pytest
import torch

import oracle
from gated_delta_rule_spec_gb300 import binding
from gated_delta_rule_spec_gb300 import inputs as gen
from tests.harness import Scenario, to_dev, to_host

pytestmark = pytest.mark.gpu


@pytest.fixture
def zero_wait_limit():
    prev = binding.set_wait_limit(0)
    try:
        yield
    finally:
        binding.set_wait_limit(binding.WAIT_LIMIT_DEFAULT)
    assert prev == (1 << 20)


def test_verify_tile_wait_runs_out_then_recovers():
    wl = gen.Workload("timeout-verify", B=4, H=2, HV=4, K=128, V=128, T=4, L=16, prefix=16)
    sc = Scenario(wl, B=4, seed=101, num_slots=6, random_cursors=True)
    assert binding.verify_path(sc.layer) == "tc"
    w = sc.window()
    dev = {n: to_dev(x) for n, x in w.items()}
    prev = binding.set_wait_limit(0)
    try:
        binding.verify(sc.layer, sc.cur, sc.slot_dev, dev["q"], dev["k"], dev["v"], dev["a"],
                       dev["b"], sc.A_log_dev, sc.dt_bias_dev)
        st = binding.read_status(sc.cur)
    finally:
        binding.set_wait_limit(binding.WAIT_LIMIT_DEFAULT)
    assert prev == 1 << 20
    assert st & binding.ST_TIMEOUT
    # the same call again, normal limit: the oracle's single verify of this window
    out, o_orc, st2 = sc.verify(w)
    assert st2 == 0 and binding.read_status(sc.cur) == 0
    assert sc.out_error(out, o_orc) <= sc.out_tol()
    sc.check_ring()
    sc.check_cursors()


def test_fold_wait_runs_out_poisons_its_rows_only(zero_wait_limit):
    wl = gen.Workload("timeout-fold", B=6, H=2, HV=4, K=128, V=128, T=4, L=16, prefix=16)
    n = 9
    rng = gen.rng_for(111, "timeout-fold")
    wp, base, flag = gen.random_cursors(rng, n, wl.L, wl.T)
    wp[:] = 7
    sc = Scenario(wl, B=6, seed=111, num_slots=n, slot_idx=np.array([4, 0, 7, -1, 2, 5], np.int32),
                  cursors=(wp, base, flag))
    flagged_rows = [4, 7, 5]                # is_flush set for three of the batch's slots
    flag_dev = np.zeros(n, np.int32)
    flag_dev[flagged_rows] = 1
    sc.cur.is_flush.copy_(to_dev(flag_dev))
    ck0 = sc.layer.checkpoint.clone()
    cur0 = {c: to_host(getattr(sc.cur, c)).copy() for c in ("write_pos", "cache_base", "is_flush")}
    binding.fold(sc.layer, sc.cur, sc.slot_dev)
    assert binding.read_status(sc.cur) & binding.ST_TIMEOUT
    wp1, base1, fl1 = (to_host(getattr(sc.cur, c)) for c in ("write_pos", "cache_base", "is_flush"))
    for s in range(n):
        if s in flagged_rows:
            assert wp1[s] == -1 and fl1[s] == 0 and base1[s] == cur0["cache_base"][s], s
        else:
            assert wp1[s] == cur0["write_pos"][s] and fl1[s] == cur0["is_flush"][s], s
            assert base1[s] == cur0["cache_base"][s]
    others = [s for s in range(n) if s not in flagged_rows]
    assert torch.equal(sc.layer.checkpoint[others].view(torch.int32), ck0[others].view(torch.int32))

    # default limit again: poisoned rows are reported and skipped by every call
    binding.set_wait_limit(binding.WAIT_LIMIT_DEFAULT)
    w = sc.window()
    dev = {k: to_dev(x) for k, x in w.items()}
    out = binding.verify(sc.layer, sc.cur, sc.slot_dev, dev["q"], dev["k"], dev["v"], dev["a"],
                         dev["b"], sc.A_log_dev, sc.dt_bias_dev)
    assert binding.read_status(sc.cur) == binding.ST_CURSOR_CORRUPT
    host = to_host(out)
    for i, s in enumerate(sc.slot_idx):
        if s in flagged_rows:
            assert not host[i].any()
    binding.commit(sc.cur, wl.T, wl.L, sc.slot_dev, to_dev(np.ones(sc.B, np.int32)))
    assert binding.read_status(sc.cur) == binding.ST_CURSOR_CORRUPT
    assert all(to_host(sc.cur.write_pos)[s] == -1 for s in flagged_rows)

    # reset + prefill rebuild them; decode then matches the oracle again
    binding.reset(sc.cur, sc.slot_dev)
    oracle.reset(sc.dims, sc.orc_cur, sc.slot_idx)
    sc.check_cursors()
    N = 8
    pw = gen.window_inputs(sc.rng, sc.B, N, wl.H, wl.HV, wl.K, wl.V, wl.io_dtype)
    pdev = {k: to_dev(x) for k, x in pw.items()}
    binding.prefill(sc.layer, sc.cur, sc.slot_dev, pdev["q"], pdev["k"], pdev["v"], pdev["a"],
                    pdev["b"], sc.A_log_dev, sc.dt_bias_dev, from_zero=True)
    f = {k: gen.to_f64(x) for k, x in pw.items()}
    _, st = oracle.prefill(sc.dims, sc.orc, sc.orc_cur, sc.slot_idx, f["q"], f["k"], f["v"], f["a"],
                           f["b"], sc.A_log, sc.dt_bias, from_zero=True)
    assert st == 0 and binding.read_status(sc.cur) == 0
    sc.check_cursors()
    out, o_orc, st = sc.verify(sc.window())
    assert st == 0 and sc.out_error(out, o_orc) <= sc.out_tol()
    assert binding.read_status(sc.cur) == 0
