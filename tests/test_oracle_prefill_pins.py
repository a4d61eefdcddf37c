"""Pins of the oracle's prefill against things other than itself.

Prefill runs the GDN recurrence over a row's prompt tokens, reads out every
token, keeps the final state as the checkpoint and resets the row's cursors
(the prefill -> decode handoff of the blog post on sglang PR #28695,
appendix A.2).  Here it is checked against the recurrence written as dense
matrices with numpy, against its own chunking (two calls equal one), and for
its cursor and status rules.  No GPU is needed.
"""
import math

import numpy as np
import pytest

import oracle
from gated_delta_rule_spec_gb300 import inputs as gen


def _softplus(x):
    return x if x > 20.0 else math.log1p(math.exp(x))


def _dense_prefill(d, S0, q, k, v, a, b, A_log, dt_bias, per_key):
    """Dense-matrix recurrence of one (row, v-head): returns (outputs [N, V], S_N)."""
    S = S0.copy()
    outs = []
    for t in range(q.shape[0]):
        kh = k[t] / math.sqrt(float(k[t] @ k[t]) + d.l2_eps)
        qh = q[t] / math.sqrt(float(q[t] @ q[t]) + d.l2_eps)
        beta = 1.0 / (1.0 + math.exp(-b[t]))
        P = np.eye(d.K) - beta * np.outer(kh, kh)
        if per_key:
            g = np.array([-math.exp(A_log) * _softplus(a[t][j] + dt_bias[j]) for j in range(d.K)])
            S = S @ np.diag(np.exp(g)) @ P + beta * np.outer(v[t], kh)
        else:
            g = -math.exp(A_log) * _softplus(a[t] + dt_bias)
            S = math.exp(g) * S @ P + beta * np.outer(v[t], kh)
        outs.append(d.scale * S @ qh)
    return np.array(outs), S


def _inputs(rng, d, B, N):
    w = gen.window_inputs(rng, B, N, d.H, d.HV, d.K, d.V, gen.FP32, d.per_key_gate)
    A_log, dt_bias = gen.layer_params(rng, d.HV, d.K, d.per_key_gate)
    return ({n: gen.to_f64(x) for n, x in w.items()}, A_log.astype(np.float64),
            dt_bias.astype(np.float64))


def _layer(rng, d):
    ring = gen.garbage_ring(rng, d.num_slots, d.H, d.HV, d.L, d.K, d.V, gen.FP32, d.per_key_gate)
    return oracle.Layer(d, checkpoint=rng.normal(size=(d.num_slots, d.HV, d.V, d.K)) * 0.5,
                        rawv=gen.to_f64(ring["rawv"]), rawk=gen.to_f64(ring["rawk"]),
                        ring_g=-np.abs(ring["g"].astype(np.float64)),
                        ring_beta=np.full(ring["beta"].shape, 0.5))


@pytest.mark.parametrize("per_key", [False, True])
@pytest.mark.parametrize("from_zero", [True, False])
def test_prefill_equals_dense_recurrence(per_key, from_zero):
    d = oracle.Dims(H=2, HV=4, K=6, V=5, T=2, L=8, num_slots=4, per_key_gate=per_key, scale=0.7)
    rng = np.random.default_rng(31 + 2 * per_key + from_zero)
    ly = _layer(rng, d)
    ck0 = ly.checkpoint.copy()
    B, N = 2, 7
    slots = np.array([3, 1], np.int32)
    cur = oracle.Cursors(d.num_slots, np.zeros(4, np.int32), np.array([5, 2, 0, 7], np.int32),
                         np.array([0, 1, 0, 1], np.int32))
    w, A_log, dt = _inputs(rng, d, B, N)
    out, st = oracle.prefill(d, ly, cur, slots, w["q"], w["k"], w["v"], w["a"], w["b"], A_log, dt,
                             from_zero=from_zero)
    assert st == 0
    G = d.HV // d.H
    for bb, slot in enumerate(slots):
        for hv in range(d.HV):
            S0 = np.zeros((d.V, d.K)) if from_zero else ck0[slot, hv]
            a = w["a"][bb, :, hv]
            dtb = dt[hv]
            o_ref, S_ref = _dense_prefill(d, S0, w["q"][bb, :, hv // G], w["k"][bb, :, hv // G],
                                          w["v"][bb, :, hv], a, w["b"][bb, :, hv], A_log[hv], dtb,
                                          per_key)
            np.testing.assert_allclose(out[bb, :, hv], o_ref, rtol=1e-11, atol=1e-12)
            np.testing.assert_allclose(ly.checkpoint[slot, hv], S_ref, rtol=1e-11, atol=1e-12)
    # the batch's slots (3, 1) have their cursors reset for decode; slots 0 and
    # 2 are not in the batch and keep cursors and checkpoint
    assert list(cur.write_pos) == [0, 0, 0, 0]
    assert list(cur.cache_base) == [5, 0, 0, 0]
    assert list(cur.is_flush) == [0, 0, 0, 0]
    for s in (0, 2):
        assert np.array_equal(ly.checkpoint[s], ck0[s])


def test_prefill_in_two_calls_equals_one_call_bitwise():
    """Chunked prefill: N1 tokens from zero, then N2 tokens from the checkpoint,
    gives the same bits as N1 + N2 tokens in one call."""
    d = oracle.Dims(H=2, HV=2, K=8, V=4, T=2, L=8, num_slots=2)
    rng = np.random.default_rng(41)
    B, N1, N2 = 2, 5, 4
    slots = np.array([0, 1], np.int32)
    w, A_log, dt = _inputs(rng, d, B, N1 + N2)
    ly1, ly2 = _layer(rng, d), _layer(rng, d)
    c1, c2 = oracle.Cursors(2), oracle.Cursors(2)
    out_all, st = oracle.prefill(d, ly1, c1, slots, *(w[n] for n in ("q", "k", "v", "a", "b")),
                                 A_log, dt)
    assert st == 0
    part = lambda lo, hi: [w[n][:, lo:hi] for n in ("q", "k", "v", "a", "b")]  # noqa: E731
    o1, _ = oracle.prefill(d, ly2, c2, slots, *part(0, N1), A_log, dt)
    o2, _ = oracle.prefill(d, ly2, c2, slots, *part(N1, N1 + N2), A_log, dt, from_zero=False)
    assert np.array_equal(np.concatenate([o1, o2], axis=1), out_all)
    assert np.array_equal(ly1.checkpoint, ly2.checkpoint)


def test_prefill_status_padding_and_unfolded_rows():
    d = oracle.Dims(H=1, HV=1, K=4, V=3, T=2, L=8, num_slots=3)
    rng = np.random.default_rng(51)
    ly = _layer(rng, d)
    ck0 = ly.checkpoint.copy()
    w, A_log, dt = _inputs(rng, d, 4, 3)
    slots = np.array([-1, 7, 1, 2], np.int32)     # padding, out of range, unfolded, fine
    cur = oracle.Cursors(3, np.array([0, 5, 0], np.int32), np.array([0, 3, 4], np.int32),
                         np.array([0, 0, 0], np.int32))
    out, st = oracle.prefill(d, ly, cur, slots, w["q"], w["k"], w["v"], w["a"], w["b"], A_log, dt,
                             from_zero=False)
    assert st == oracle.ST_SLOT_OOR | oracle.ST_UNFOLDED
    assert not out[:3].any()                      # skipped rows read out zeros
    assert out[3].any()
    assert np.array_equal(ly.checkpoint[1], ck0[1])   # the unfolded slot is untouched
    assert (cur.write_pos[1], cur.cache_base[1]) == (5, 3)
    assert (cur.write_pos[2], cur.cache_base[2]) == (0, 0)
