"""Pins of the oracle's snapshot variant (the per-draft snapshot design that
the ReplaySSM ring replaces, kept as a comparison) against the recurrence
written as dense matrices, and of its commit.  No GPU is needed.
"""
import numpy as np
import pytest

import oracle
from tests.test_oracle_prefill_pins import _dense_prefill, _inputs, _layer


@pytest.mark.parametrize("per_key", [False, True])
def test_snapshot_verify_equals_dense_recurrence(per_key):
    d = oracle.Dims(H=2, HV=4, K=6, V=5, T=3, L=8, num_slots=4, per_key_gate=per_key, scale=0.8)
    rng = np.random.default_rng(71 + per_key)
    ly = _layer(rng, d)
    ck0 = ly.checkpoint.copy()
    slots = np.array([2, -1, 0], np.int32)
    w, A_log, dt = _inputs(rng, d, 3, d.T)
    out, snap, st = oracle.snapshot_verify(d, ly, slots, w["q"], w["k"], w["v"], w["a"], w["b"],
                                           A_log, dt)
    assert st == 0
    assert np.array_equal(ly.checkpoint, ck0)     # verify only reads the state
    assert not out[1].any() and not snap[1].any()  # padding row
    G = d.HV // d.H
    for bb in (0, 2):
        slot = slots[bb]
        for hv in range(d.HV):
            for s in range(d.T):
                o_ref, S_ref = _dense_prefill(d, ck0[slot, hv], w["q"][bb, :s + 1, hv // G],
                                              w["k"][bb, :s + 1, hv // G], w["v"][bb, :s + 1, hv],
                                              w["a"][bb, :s + 1, hv], w["b"][bb, :s + 1, hv],
                                              A_log[hv], dt[hv], per_key)
                np.testing.assert_allclose(out[bb, s, hv], o_ref[s], rtol=1e-11, atol=1e-12)
                np.testing.assert_allclose(snap[bb, s, hv], S_ref, rtol=1e-11, atol=1e-12)


def test_snapshot_commit_copies_the_accepted_state():
    d = oracle.Dims(H=1, HV=2, K=4, V=3, T=3, L=8, num_slots=4)
    rng = np.random.default_rng(81)
    ly = _layer(rng, d)
    ck0 = ly.checkpoint.copy()
    slots = np.array([3, 1, 0, 9, -1], np.int32)
    snap = rng.normal(size=(5, d.T, d.HV, d.V, d.K))
    acc = np.array([2, 0, 3, 1, 1], np.int32)
    assert oracle.snapshot_commit(d, ly, slots, acc, snap) == oracle.ST_SLOT_OOR
    assert np.array_equal(ly.checkpoint[3], snap[0, 1])
    assert np.array_equal(ly.checkpoint[1], ck0[1])      # accept_len 0 keeps the state
    assert np.array_equal(ly.checkpoint[0], snap[2, 2])
    assert np.array_equal(ly.checkpoint[2], ck0[2])      # not in the batch
    bad = np.array([4, 0, 0, 0, 0], np.int32)
    assert oracle.snapshot_commit(d, ly, slots, bad, snap) & oracle.ST_ACCEPT_RANGE


def test_snapshot_and_ring_agree_on_outputs_and_committed_state():
    """The comparison is fair: from the same state the snapshot path and the
    ring path (verify, commit, fold) give the same outputs and, after the
    commit, the same state."""
    d = oracle.Dims(H=2, HV=2, K=8, V=4, T=4, L=8, num_slots=2)
    rng = np.random.default_rng(91)
    ring_ly, snap_ly = _layer(rng, d), None
    snap_ly = oracle.Layer(d, checkpoint=ring_ly.checkpoint.copy(), rawv=ring_ly.rawv.copy(),
                           rawk=ring_ly.rawk.copy(), ring_g=ring_ly.ring_g.copy(),
                           ring_beta=ring_ly.ring_beta.copy())
    slots = np.array([1, 0], np.int32)
    cur = oracle.Cursors(2)                       # empty ring: W = 0
    w, A_log, dt = _inputs(rng, d, 2, d.T)
    o_ring, st = oracle.verify(d, ring_ly, cur, slots, w["q"], w["k"], w["v"], w["a"], w["b"], A_log, dt)
    o_snap, snap, st2 = oracle.snapshot_verify(d, snap_ly, slots, w["q"], w["k"], w["v"], w["a"],
                                               w["b"], A_log, dt)
    assert st == st2 == 0
    np.testing.assert_allclose(o_ring, o_snap, rtol=1e-10, atol=1e-12)
    acc = np.array([3, 4], np.int32)
    assert oracle.commit(d, cur, slots, acc) == 0
    cur.is_flush[:] = 1                            # fold now, whatever the margin
    assert oracle.fold(d, ring_ly, cur, slots) == 0
    assert oracle.snapshot_commit(d, snap_ly, slots, acc, snap) == 0
    np.testing.assert_allclose(ring_ly.checkpoint, snap_ly.checkpoint, rtol=1e-12, atol=1e-13)
