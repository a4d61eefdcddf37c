"""GPU checks of the state the calls leave behind, against the fp64 oracle.

* The tensor-core verify and the fold with raw (non-unit) q, k and ring-history
  keys: every key and query row scaled by a factor in [0.25, 4], so a kernel
  that skipped its L2 norm would be far off.
* gdn_spec_reset against the oracle's reset, bitwise, with padding rows and a
  slot out of range, over a scattered pool.
* gdn_spec_fold of three layers in one call (and of fifty, more than one
  launch takes) against the oracle's fold of the same layers.
* Bitwise "untouched": verify leaves every checkpoint and the cursors as they
  were; fold leaves the checkpoint of every slot it did not fold as it was;
  commit skips rows with corrupt cursors and reports them.
* A fold over more batch rows than its flag scan takes in one pass.

All through the C ABI.  Bars as elsewhere: outputs max-abs <= 3e-2 (bf16 I/O),
each folded (slot, v-head) checkpoint within 1e-3 relative Frobenius error,
cursors bit-exact.
"""
import numpy as np
import pytest
import torch

import oracle
from gated_delta_rule_spec_gb300 import binding
from gated_delta_rule_spec_gb300 import inputs as gen
from tests.harness import CKPT_REL_FRO, Scenario, to_host

pytestmark = pytest.mark.gpu
WL = gen.WORKLOADS


def _flagged(sc):
    f = to_host(sc.cur.is_flush)
    return sorted(int(s) for s in sc.slot_idx if s >= 0 and f[s])


def test_tc_raw_q_k_and_history_keys_with_folds():
    """Qwen3-Next shape on the tensor-core path; prefix, ring history and every
    window's q and k rows scaled by factors in [0.25, 4]; several rounds with
    folds, so the fold's key norm runs too."""
    wl = WL["C2"]
    sc = Scenario(wl, B=8, seed=51, num_slots=24, random_cursors=True, key_scale=(0.25, 4.0))
    assert binding.verify_path(sc.layer) == "tc"
    # the inputs really are far from unit norm
    w = sc.window()
    norms = np.linalg.norm(gen.to_f64(w["k"]), axis=-1)
    assert norms.min() < 0.4 and norms.max() > 2.5
    folded = 0
    for r in range(12):
        if r:
            w = sc.window()
        out, o_orc, st = sc.verify(w)
        assert st == 0
        err = sc.out_error(out, o_orc)
        assert err <= sc.out_tol(), f"round {r}: output error {err}"
        sc.check_ring()
        acc = gen.accept_lens(sc.rng, sc.B, wl.T, full_frac=0.5)
        assert sc.commit(acc) == 0
        flagged = _flagged(sc)
        folded += len(flagged)
        assert sc.fold() == 0
        sc.check_cursors()
        used = sorted(set(sc.slot_idx.tolist()))
        e = sc.ckpt_error_per_slot(used)
        assert e <= CKPT_REL_FRO, f"round {r}: checkpoint error {e}"
    assert folded > 0
    assert binding.read_status(sc.cur) == 0


def test_reset_matches_oracle_bitwise():
    """Random cursors over a 64-slot pool; reset names scattered slots, two
    padding rows and one slot past the pool.  All three cursor arrays must
    equal the oracle's, bitwise (so slots not named are untouched), and the
    status must say SLOT_OOR."""
    wl = gen.Workload("reset", B=10, H=2, HV=4, K=32, V=32, T=4, L=16, prefix=0)
    rng = gen.rng_for(61, "reset")
    n = 64
    wp, base, _ = gen.random_cursors(rng, n, wl.L, wl.T)
    flag = rng.integers(0, 2, size=n).astype(np.int32)
    slots = gen.scattered_slots(rng, n, 7)
    slot_idx = np.concatenate([slots[:3], [-1], slots[3:], [-5, n + 3]]).astype(np.int32)
    sc = Scenario(wl, B=len(slot_idx), seed=61, num_slots=n, slot_idx=slot_idx,
                  cursors=(wp, base, flag))
    before = {c: to_host(getattr(sc.cur, c)).copy() for c in ("write_pos", "cache_base", "is_flush")}
    binding.reset(sc.cur, sc.slot_dev)
    st = oracle.reset(sc.dims, sc.orc_cur, sc.slot_idx)
    assert st == oracle.ST_SLOT_OOR
    assert binding.read_status(sc.cur) == st
    sc.check_cursors()
    named = set(int(s) for s in slots)
    for c, arr in before.items():
        got = to_host(getattr(sc.cur, c))
        for s in range(n):
            if s in named:
                assert got[s] == 0, (c, s)
            else:
                assert got[s] == arr[s], (c, s)


def _layers_sharing_cursors(n_layers, wl, B, num_slots, seed, cursors=None, **kw):
    """n_layers Scenarios with the same slots and the same cursors (each with its
    own checkpoint and ring history at those cursors); every layer then uses
    layer 0's device and oracle cursor objects."""
    rng = gen.rng_for(seed, "layers", n_layers)
    if cursors is None:
        cursors = gen.random_cursors(rng, num_slots, wl.L, wl.T)
    slots = gen.scattered_slots(rng, num_slots, B)
    scs = [Scenario(wl, B=B, seed=seed + 7 * i, num_slots=num_slots, slot_idx=slots,
                    cursors=cursors, **kw) for i in range(n_layers)]
    for sc in scs[1:]:
        sc.cur, sc.orc_cur = scs[0].cur, scs[0].orc_cur
    return scs


def _fold_layers_and_compare(scs):
    s0 = scs[0]
    binding.fold([sc.layer for sc in scs], s0.cur, s0.slot_dev)
    st = oracle.fold(s0.dims, [sc.orc for sc in scs], s0.orc_cur, s0.slot_idx)
    assert st == 0
    assert binding.read_status(s0.cur) == 0
    s0.check_cursors()
    used = sorted(set(int(s) for s in s0.slot_idx if s >= 0))
    for i, sc in enumerate(scs):
        e = sc.ckpt_error_per_slot(used)
        assert e <= CKPT_REL_FRO, f"layer {i}: checkpoint error {e}"
        # slots outside the batch keep their bytes
        unused = sorted(set(range(sc.num_slots)) - set(used))
        got = to_host(sc.layer.checkpoint)[unused]
        assert np.array_equal(got, sc.orc.checkpoint[unused].astype(np.float32)), f"layer {i}"


def test_fold_three_layers_in_one_call():
    """Three layers with different checkpoints and rings, one set of cursors:
    verify each layer, commit once, fold all three in one call.  Each layer's
    checkpoint must match the oracle's fold of the same three layers, and the
    cursors must move once."""
    wl = gen.Workload("three-layers", B=6, H=2, HV=4, K=128, V=128, T=4, L=16, prefix=16)
    scs = _layers_sharing_cursors(3, wl, B=6, num_slots=10, seed=71, decay_shift=1.0)
    assert binding.verify_path(scs[0].layer) == "tc"
    s0 = scs[0]
    for rnd in range(4):
        for sc in scs:   # each layer's verify reads the shared cursors
            out, o_orc, st = sc.verify(sc.window())
            assert st == 0 and sc.out_error(out, o_orc) <= sc.out_tol()
            sc.check_ring()
        acc = gen.accept_lens(s0.rng, s0.B, wl.T, full_frac=0.6)
        assert s0.commit(acc) == 0
        s0.check_cursors()
        _fold_layers_and_compare(scs)


def test_fold_fifty_layers_more_than_one_launch():
    """Fifty small layers folded in one call (the library folds at most 48
    layers per launch, so this takes two) against the oracle."""
    wl = gen.Workload("fifty-layers", B=3, H=1, HV=2, K=32, V=32, T=2, L=8, prefix=4)
    # every slot flagged, its ring holding write_pos committed records
    cursors = (np.array([6, 7, 5, 8, 6], np.int32), np.array([3, 0, 7, 5, 1], np.int32),
               np.ones(5, np.int32))
    scs = _layers_sharing_cursors(50, wl, B=3, num_slots=5, seed=81, cursors=cursors)
    _fold_layers_and_compare(scs)


def test_verify_and_fold_leave_other_state_bitwise_untouched():
    """B = 32 rows of a 512-slot pool at the Qwen3-Next shape: verify leaves
    the whole checkpoint pool and all cursors bitwise unchanged; after commit,
    fold leaves the checkpoint of every slot it did not fold (not flagged, or
    not in the batch) bitwise unchanged."""
    wl = WL["C2"]
    rng = gen.rng_for(91, "untouched")
    n = 512
    wp, base, flag = gen.random_cursors(rng, n, wl.L, wl.T)
    wp[::2] = wl.L - 2 * wl.T          # half the pool at the margin: any accept flags it
    sc = Scenario(wl, B=32, seed=91, num_slots=n, cursors=(wp, base, flag))
    ck0 = sc.layer.checkpoint.clone()
    cur0 = {c: getattr(sc.cur, c).clone() for c in ("write_pos", "cache_base", "is_flush")}
    out, o_orc, st = sc.verify(sc.window())
    assert st == 0 and sc.out_error(out, o_orc) <= sc.out_tol()
    assert torch.equal(sc.layer.checkpoint.view(torch.int32), ck0.view(torch.int32))
    for c, t in cur0.items():
        assert torch.equal(getattr(sc.cur, c), t), c
    acc = gen.accept_lens(sc.rng, sc.B, wl.T)
    assert sc.commit(acc) == 0
    sc.check_cursors()
    flagged = _flagged(sc)
    assert 0 < len(flagged) < sc.B
    ck1 = to_host(sc.layer.checkpoint).copy()
    assert sc.fold() == 0
    sc.check_cursors()
    ck2 = to_host(sc.layer.checkpoint)
    untouched = sorted(set(range(sc.num_slots)) - set(flagged))
    assert np.array_equal(ck2[untouched].view(np.uint32), ck1[untouched].view(np.uint32))
    assert sc.ckpt_error_per_slot(flagged) <= CKPT_REL_FRO
    assert binding.read_status(sc.cur) == 0


def test_commit_rejects_corrupt_cursors_like_the_oracle():
    wl = gen.Workload("commit-corrupt", B=6, H=1, HV=2, K=32, V=32, T=4, L=16, prefix=0)
    n = 8
    wp = np.array([-1, 17, 3, 16, 2, 5, 0, 9], np.int32)
    base = np.array([0, 0, 16, 15, -2, 3, 7, 1], np.int32)
    flag = np.array([0, 0, 0, 1, 0, 0, 0, 0], np.int32)
    sc = Scenario(wl, B=6, seed=3, num_slots=n, slot_idx=np.arange(6, dtype=np.int32),
                  cursors=(wp, base, flag))
    st = sc.commit(np.array([1, 1, 1, 0, 1, 2], np.int32))
    assert st == oracle.ST_CURSOR_CORRUPT
    assert binding.read_status(sc.cur) == st
    sc.check_cursors()


def test_fold_more_rows_than_one_scan_pass():
    """B = 300 rows, more than the fold's flag scan takes in one pass (256 rows
    with the scalar gate): rows of both passes are flagged and folded in the
    same launch.  L = 16, so most rows fold every few rounds; cursors bit-exact
    after every call, every used slot's checkpoint within the bar."""
    wl = gen.Workload("fold-300", B=300, H=1, HV=2, K=128, V=128, T=4, L=16, prefix=8)
    sc = Scenario(wl, B=300, seed=81, num_slots=320, random_cursors=True)
    assert binding.verify_path(sc.layer) == "tc"
    folded_late = 0
    for r in range(6):
        out, o_orc, st = sc.verify(sc.window())
        assert st == 0 and sc.out_error(out, o_orc) <= sc.out_tol(), f"round {r}"
        acc = gen.accept_lens(sc.rng, sc.B, wl.T, full_frac=0.6)
        assert sc.commit(acc) == 0
        sc.check_cursors()
        flagged_rows = [i for i, s in enumerate(sc.slot_idx) if s >= 0 and sc.orc_cur.is_flush[s]]
        folded_late += sum(1 for i in flagged_rows if i >= 256)
        assert sc.fold() == 0
        sc.check_cursors()
    assert folded_late > 0
    used = sorted(set(int(s) for s in sc.slot_idx if s >= 0))
    assert sc.ckpt_error_per_slot(used) <= CKPT_REL_FRO
