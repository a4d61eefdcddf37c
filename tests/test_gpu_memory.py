"""The ring path allocates no per-draft state: device free memory is the same
before and after verify -> commit -> fold steps at the Qwen3-Next shape, B = 128
(a [B, T, HV, V, K] fp32 snapshot there would be 1 GiB)."""
import numpy as np
import pytest
import torch

from gated_delta_rule_spec_gb300 import binding
from gated_delta_rule_spec_gb300 import inputs as gen

pytestmark = pytest.mark.gpu


def test_verify_commit_fold_allocate_nothing():
    B, H, HV, K, V, T, L, slots_n = 128, 16, 32, 128, 128, 4, 64, 160
    rng = gen.rng_for(5, "memory", B)
    layer = binding.SpecLayer(H, HV, K, V, T, L, slots_n)
    cur = binding.SpecCursors(slots_n)
    A_log, dt_bias = (torch.from_numpy(x).cuda() for x in gen.layer_params(rng, HV, K, False))
    slots = torch.from_numpy(gen.scattered_slots(rng, slots_n, B)).cuda()
    wins = [{n: torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).cuda()
             for n, x in gen.window_inputs(rng, B, T, H, HV, K, V, gen.BF16).items()} for _ in range(3)]
    accs = [torch.from_numpy(gen.accept_lens(rng, B, T)).cuda() for _ in range(3)]
    out = torch.empty(B, T, HV, V, dtype=torch.bfloat16, device="cuda")

    def step(i):
        w = wins[i % 3]
        binding.verify(layer, cur, slots, w["q"], w["k"], w["v"], w["a"], w["b"], A_log, dt_bias, out=out)
        binding.commit(cur, T, L, slots, accs[i % 3])
        binding.fold(layer, cur, slots)

    step(0)                      # modules loaded, attributes set
    torch.cuda.synchronize()
    free0, total = torch.cuda.mem_get_info()
    snapshot_bytes = B * T * HV * V * K * 4
    for i in range(1, 40):
        step(i)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free0 - free1 < 16 << 20, (free0, free1)
    assert snapshot_bytes == 1 << 30
    assert binding.read_status(cur) == 0
