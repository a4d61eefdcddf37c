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


def _verify_from_d_ring(d, ly, dring, cur, slot, hv, w, bb, A_log, dtb):
    """One (row, v-head) unit of a verify that takes the history through the
    cached deltas (the derived-d design): only the T x T window system is
    solved.  Written here with dense numpy, independently of the oracle."""
    T, L, V = d.T, d.L, d.V
    h = hv // (d.HV // d.H)
    base, W = cur.cache_base[slot], cur.write_pos[slot]
    pos = [(base + o) % L for o in range(W)]
    kh = [_khat(ly.rawk[slot, h, p]) for p in pos]
    dh = [dring[slot, hv, p] for p in pos]
    kw = [_khat(w["k"][bb, s, h]) for s in range(T)]
    qw = [_khat(w["q"][bb, s, h]) for s in range(T)]
    gw, bw = oracle.gate(A_log[hv:hv + 1], w["a"][bb, :, hv:hv + 1], dtb[hv:hv + 1],
                         w["b"][bb, :, hv:hv + 1])
    gw, bw = gw.reshape(-1), bw.reshape(-1)
    cum = np.concatenate([[0.0], np.cumsum([ly.ring_g[slot, hv, p] for p in pos] + list(gw))])

    def gam(i, r):   # decay over tokens r+1..i (r = -1: from the checkpoint)
        return np.exp(cum[i + 1] - cum[r + 1])

    S0 = ly.checkpoint[slot, hv]
    Hk = [sum((gam(W + s, r) * (kh[r] @ kw[s]) * dh[r] for r in range(W)), np.zeros(V)) for s in range(T)]
    Hq = [sum((gam(W + s, r) * (kh[r] @ qw[s]) * dh[r] for r in range(W)), np.zeros(V)) for s in range(T)]
    R = np.array([bw[s] * (w["v"][bb, s, hv] - gam(W + s, -1) * (S0 @ kw[s]) - Hk[s]) for s in range(T)])
    A = np.array([[bw[s] * gam(W + s, W + s2) * (kw[s2] @ kw[s]) if s2 < s else 0.0
                   for s2 in range(T)] for s in range(T)])
    Dw = np.linalg.solve(np.eye(T) + A, R)
    out = np.array([d.scale * (gam(W + s, -1) * (S0 @ qw[s]) + Hq[s] +
                               sum(gam(W + s, W + s2) * (kw[s2] @ qw[s]) * Dw[s2] for s2 in range(s + 1)))
                    for s in range(T)])
    return out, Dw


def test_cached_deltas_reproduce_verify_over_rounds_with_folds():
    """Keep the window d's that verify_d returns in a ring (at the window's ring
    positions, as the raw records are kept), then verify -> commit -> fold for
    many rounds: a verify that takes its history through those d's alone gives
    the oracle's outputs and window d's.  Pins verify_d's deltas as the ones a
    derived-d ring holds, across rejected drafts and folds."""
    from gated_delta_rule_spec_gb300 import inputs as gen
    rng = np.random.default_rng(3)
    d = oracle.Dims(H=2, HV=4, K=16, V=8, T=4, L=16, num_slots=3, scale=0.9)
    ly = oracle.Layer(d, checkpoint=rng.standard_normal((3, d.HV, d.V, d.K)) * 0.3)
    dring = np.zeros((3, d.HV, d.L, d.V))
    cur = oracle.Cursors(3)
    slots = np.array([2, 0], np.int32)
    A_log, dtb = (x.astype(np.float64) for x in gen.layer_params(rng, d.HV, d.K, False))
    folds = 0
    for _ in range(30):
        w = {n: gen.to_f64(x) for n, x in
             gen.window_inputs(rng, 2, d.T, d.H, d.HV, d.K, d.V, gen.BF16).items()}
        w["a"] = w["a"] - 2.0
        before, cur0 = ly.copy(), cur.copy()
        o_orc, d_orc, st = oracle.verify_d(d, ly, cur, slots, w["q"], w["k"], w["v"], w["a"],
                                           w["b"], A_log, dtb)
        assert st == 0
        for bb, slot in enumerate(slots):
            for hv in range(d.HV):
                o, dw = _verify_from_d_ring(d, before, dring, cur0, slot, hv, w, bb, A_log, dtb)
                np.testing.assert_allclose(o, o_orc[bb, :, hv], rtol=1e-9, atol=1e-11)
                np.testing.assert_allclose(dw, d_orc[bb, :, hv], rtol=1e-9, atol=1e-11)
                for s in range(d.T):
                    dring[slot, hv, (cur0.cache_base[slot] + cur0.write_pos[slot] + s) % d.L] = dw[s]
        assert oracle.commit(d, cur, slots, gen.accept_lens(rng, 2, d.T)) == 0
        folds += int(cur.is_flush[slots].sum())
        assert oracle.fold(d, ly, cur, slots) == 0
    assert folds > 0
