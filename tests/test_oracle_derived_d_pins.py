"""Pins of the oracle's corrected deltas (verify_d), the values a ring that
caches d instead of raw v (the derived-d design) would hold.  No GPU is needed.

d_t = beta_t (v_t - S k^_t), with S the state decayed by token t's gate (blog
post on sglang PR #28695, §12.1).  It is pinned three ways against things other
than the oracle:
* the closed-form UT transform: D = (I + A)^{-1} R, whose window rows are d;
* the rank-1 identity of a dense recurrence: S_t - decay_t(S_{t-1}) = d_t k^_t^T;
* reconstruction: the state after n tokens is the decayed checkpoint plus
  sum_j (decayed d_j k^_j^T), which is what a derived-d verify would rely on.
"""
import numpy as np
import pytest

import oracle
from tests.test_oracle_pins import _khat, _random_layer, _ut_closed_form, _window


def _dense_states(d, S0, ks, vs, gs, bs, per_key):
    """States after each token by the dense formula, written with matrices:
    S_t = D_t(S_{t-1}) (I - b k^ k^T) + b v k^T, D_t the decay (scalar or per key
    channel).  Returns the list [S_0 .. S_n] and the decayed predecessors."""
    K = d.K
    S = [np.array(S0, float)]
    decayed = []
    for k, v, g, b in zip(ks, vs, gs, bs):
        kh = _khat(np.asarray(k))
        Dg = np.diag(np.exp(np.broadcast_to(np.asarray(g, float), (K,))))
        Sd = S[-1] @ Dg if per_key else np.exp(float(np.asarray(g).ravel()[0])) * S[-1]
        decayed.append(Sd)
        S.append(Sd @ (np.eye(K) - b * np.outer(kh, kh)) + b * np.outer(np.asarray(v), kh))
    return S, decayed


def _case(per_key, W, seed):
    d = oracle.Dims(H=2, HV=4, K=6, V=5, T=4, L=16, num_slots=3, per_key_gate=per_key, scale=0.75)
    rng = np.random.default_rng(seed)
    ly = _random_layer(rng, d)
    ly.ring_g *= 0.05
    slot_idx = np.array([2, -1, 0], np.int32)
    cur = oracle.Cursors(d.num_slots, write_pos=[W, 0, W], cache_base=[0, 0, 13])
    win, A_log, dt = _window(rng, d, 3)
    win["a"] = win["a"] - 3.0
    return d, ly, cur, slot_idx, win, A_log, dt


def _unit_tokens(d, ly, cur, slot, bb, hv, win, g_win, b_win):
    G = d.HV // d.H
    h = hv // G
    base, wp = cur.cache_base[slot], cur.write_pos[slot]
    pos = [(base + o) % d.L for o in range(wp)]
    ks = [ly.rawk[slot, h, p] for p in pos] + list(win["k"][bb, :, h])
    vs = [ly.rawv[slot, hv, p] for p in pos] + list(win["v"][bb, :, hv])
    gs = [ly.ring_g[slot, hv, p] for p in pos] + list(g_win[bb, :, hv])
    bs = [ly.ring_beta[slot, hv, p] for p in pos] + list(b_win[bb, :, hv])
    return wp, ks, vs, gs, bs


@pytest.mark.parametrize("per_key", [False, True])
@pytest.mark.parametrize("W", [0, 3, 7])
def test_window_d_equals_closed_form_and_rank_one_identity(per_key, W):
    d, ly, cur, slot_idx, win, A_log, dt = _case(per_key, W, 300 + W + 10 * per_key)
    out_ref, st_ref = oracle.verify(d, ly.copy(), cur, slot_idx, win["q"], win["k"], win["v"],
                                    win["a"], win["b"], A_log, dt)
    out, dwin, st = oracle.verify_d(d, ly.copy(), cur, slot_idx, win["q"], win["k"], win["v"],
                                    win["a"], win["b"], A_log, dt)
    assert st == st_ref == 0
    assert np.array_equal(out, out_ref)          # the same outputs, bit for bit
    assert not dwin[1].any()                     # padding row
    g_win, b_win = oracle.gate(A_log, win["a"], dt, win["b"], per_key_gate=per_key)
    G = d.HV // d.H
    for bb in (0, 2):
        slot = slot_idx[bb]
        for hv in range(d.HV):
            h = hv // G
            wp, ks, vs, gs, bs = _unit_tokens(d, ly, cur, slot, bb, hv, win, g_win, b_win)
            hist = {"k": ks[:wp], "v": vs[:wp], "g": gs[:wp], "beta": bs[:wp]}
            _, (D_inv, D_neu) = _ut_closed_form(
                d, ly.checkpoint[slot, hv], hist, win["k"][bb, :, h], win["v"][bb, :, hv],
                win["q"][bb, :, h], list(g_win[bb, :, hv]), list(b_win[bb, :, hv]), with_d=True)
            np.testing.assert_allclose(dwin[bb, :, hv], D_inv[wp:], rtol=1e-9, atol=1e-11)
            np.testing.assert_allclose(dwin[bb, :, hv], D_neu[wp:], rtol=1e-9, atol=1e-11)
            S, decayed = _dense_states(d, ly.checkpoint[slot, hv], ks, vs, gs, bs, per_key)
            for s in range(d.T):
                t = wp + s
                kh = _khat(np.asarray(ks[t]))
                diff = S[t + 1] - decayed[t]
                np.testing.assert_allclose(diff, np.outer(dwin[bb, s, hv], kh), rtol=1e-10,
                                           atol=1e-12)


@pytest.mark.parametrize("per_key", [False, True])
def test_state_reconstructed_from_checkpoint_and_deltas(per_key):
    """S_n = decay(n-1, -1)(S0) + sum_j d_j (decay(n-1, j) k^_j)^T with the
    window's d from the oracle and the history's d from a dense recurrence."""
    W = 6
    d, ly, cur, slot_idx, win, A_log, dt = _case(per_key, W, 400 + per_key)
    _, dwin, st = oracle.verify_d(d, ly.copy(), cur, slot_idx, win["q"], win["k"], win["v"],
                                  win["a"], win["b"], A_log, dt)
    assert st == 0
    g_win, b_win = oracle.gate(A_log, win["a"], dt, win["b"], per_key_gate=per_key)
    K = d.K
    for bb in (0, 2):
        slot = slot_idx[bb]
        for hv in range(d.HV):
            wp, ks, vs, gs, bs = _unit_tokens(d, ly, cur, slot, bb, hv, win, g_win, b_win)
            S, decayed = _dense_states(d, ly.checkpoint[slot, hv], ks, vs, gs, bs, per_key)
            n = len(ks)
            # history deltas from the dense recurrence: its rank-1 factor, divided by
            # |k^|^2 (slightly below 1: eps sits inside the norm's square root)
            ds = []
            for t in range(wp):
                kh = _khat(np.asarray(ks[t]))
                ds.append((S[t + 1] - decayed[t]) @ kh / (kh @ kh))
            ds += [dwin[bb, s, hv] for s in range(d.T)]
            logal = np.array([np.broadcast_to(np.asarray(g, float), (K,)) for g in gs])
            rec = ly.checkpoint[slot, hv] * np.exp(logal.sum(axis=0))[None, :]
            for j in range(n):
                gam = np.exp(logal[j + 1:].sum(axis=0))        # decay from token j to the end
                rec = rec + np.outer(ds[j], _khat(np.asarray(ks[j])) * gam)
            np.testing.assert_allclose(rec, S[n], rtol=1e-10, atol=1e-12)
