"""GPU parity of the snapshot comparison variant (per-draft full states, the
design the ReplaySSM ring replaces) against the oracle: outputs, every stored
state, and the checkpoint after the commit."""
import numpy as np
import pytest
import torch

import oracle
from gated_delta_rule_spec_gb300 import binding
from gated_delta_rule_spec_gb300 import inputs as gen
from tests.harness import CKPT_REL_FRO, OUT_TOL_BF16, to_dev, to_host
from tests.test_gpu_prefill import PrefillCase

pytestmark = pytest.mark.gpu


def _rel_fro(got, ref):
    return float(np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-30))


@pytest.mark.parametrize("shape,per_key,io", [
    ((16, 32, 128, 128, 64), False, gen.BF16),
    ((16, 32, 128, 128, 64), True, gen.BF16),
    ((2, 4, 32, 40, 16), False, gen.FP32),
])
def test_snapshot_verify_and_commit(shape, per_key, io):
    H, HV, K, V, L = shape
    c = PrefillCase(H=H, HV=HV, K=K, V=V, L=L, num_slots=5, io=io, per_key=per_key, seed=101 + per_key)
    d = c.d
    slots = np.array([4, -1, 0, 2], np.int32)
    w = gen.window_inputs(c.rng, 4, d.T, H, HV, K, V, io, per_key)
    f = {n: gen.to_f64(x) for n, x in w.items()}
    o_orc, s_orc, st_orc = oracle.snapshot_verify(d, c.orc, slots, f["q"], f["k"], f["v"], f["a"], f["b"],
                                                  c.A_log.astype(np.float64), c.dt_bias.astype(np.float64))
    dev = {n: to_dev(x) for n, x in w.items()}
    out, snap = binding.snapshot_verify(c.layer, c.cur, to_dev(slots), dev["q"], dev["k"], dev["v"],
                                        dev["a"], dev["b"], torch.from_numpy(c.A_log).cuda(),
                                        torch.from_numpy(c.dt_bias).cuda())
    assert binding.read_status(c.cur) == st_orc == 0
    out_h = gen.to_f64(to_host(out))
    err = float(np.max(np.abs(out_h - o_orc)))
    assert err <= (OUT_TOL_BF16 if io == gen.BF16 else 1e-4), err
    assert not out_h[1].any()
    snap_h = to_host(snap).astype(np.float64)
    worst = max(_rel_fro(snap_h[b, s, hv], s_orc[b, s, hv])
                for b in (0, 2, 3) for s in range(d.T) for hv in range(HV))
    assert worst <= CKPT_REL_FRO, worst
    acc = np.array([3, 2, 0, 4], np.int32)
    st = oracle.snapshot_commit(d, c.orc, slots, acc, s_orc)
    binding.snapshot_commit(c.layer, c.cur, to_dev(slots), to_dev(acc), snap)
    assert binding.read_status(c.cur) == st == 0
    got = to_host(c.layer.checkpoint).astype(np.float64)
    ck = max(_rel_fro(got[s], c.orc.checkpoint[s]) for s in range(d.num_slots))
    assert ck <= CKPT_REL_FRO, ck
    print(f"snapshot {shape} per_key={per_key} {io}: output {err:.3e}, states {worst:.2e}, "
          f"checkpoint {ck:.2e}")
