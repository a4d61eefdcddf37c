"""Pins of the fp64 oracle against things other than itself.

Each test checks the oracle against mathematics the pages fix (the GDN
recurrence written as dense matrices, the closed-form chunked UT transform,
invariants and special cases, library routines for the scalar functions), so
that a dropped term, a wrong sign or index or a transposed operand in
``oracle/gdn_oracle.c`` fails here.  No GPU is needed.
"""
import itertools
import math

import numpy as np
import pytest

import oracle
from gated_delta_rule_spec_gb300 import inputs as gen

RTOL = 1e-12


def _unit(x):
    return x / np.linalg.norm(x)


def _khat(k, eps=1e-6):
    return k / math.sqrt(float(k @ k) + eps)


# --------------------------------------------------------------------- gating

def test_gate_special_values():
    # softplus above the threshold 20 is the identity
    for x in (20.0001, 25.0, 80.0, 1e4):
        assert oracle.softplus(x) == x
    # A_log = 0, a + dt_bias = 0  =>  g = -softplus(0) = -ln 2
    assert abs(oracle.gate_g(0.0, 0.0, 0.0) + math.log(2.0)) < 1e-15
    assert abs(oracle.gate_g(0.0, -0.3, 0.3) + math.log(2.0)) < 1e-15
    # sigmoid(0) = 1/2; sigmoid(-x) = 1 - sigmoid(x)
    assert oracle.gate_beta(0.0) == 0.5
    for x in (-3.0, -0.5, 0.7, 4.0):
        assert abs(oracle.gate_beta(-x) - (1.0 - oracle.gate_beta(x))) < 1e-15


def test_gate_against_library_routines():
    scipy_special = pytest.importorskip("scipy.special")
    xs = np.linspace(-30.0, 19.9, 401)
    sp = np.array([oracle.softplus(x) for x in xs])
    np.testing.assert_allclose(sp, np.logaddexp(0.0, xs), rtol=1e-14, atol=1e-300)
    bs = np.array([oracle.gate_beta(x) for x in xs])
    np.testing.assert_allclose(bs, scipy_special.expit(xs), rtol=1e-14)
    # g = -exp(A_log) * softplus(a + dt_bias)
    rng = np.random.default_rng(3)
    for _ in range(50):
        A_log, a, dt = rng.uniform(0, math.log(16)), rng.normal(), rng.uniform(-1, 1)
        want = -math.exp(A_log) * np.logaddexp(0.0, a + dt)
        assert abs(oracle.gate_g(A_log, a, dt) - want) <= 1e-14 * abs(want)


def test_gate_vectorised_kda_layout():
    rng = np.random.default_rng(4)
    HV, K = 3, 5
    A_log = rng.uniform(0, 2, HV)
    dt = rng.uniform(-1, 1, (HV, K))
    a = rng.normal(size=(2, 4, HV, K))
    b = rng.normal(size=(2, 4, HV))
    g, beta = oracle.gate(A_log, a, dt, b, per_key_gate=True)
    for i, s, hv, j in itertools.product(range(2), range(4), range(HV), range(K)):
        want = -math.exp(A_log[hv]) * np.logaddexp(0.0, a[i, s, hv, j] + dt[hv, j])
        assert abs(g[i, s, hv, j] - want) <= 1e-14 * abs(want)
    np.testing.assert_allclose(beta, 1 / (1 + np.exp(-b)), rtol=1e-14)


# --------------------------------------------------------------- L2 norm / step

def test_readout_normalises_q():
    rng = np.random.default_rng(5)
    S = rng.normal(size=(6, 8))
    q = rng.normal(size=8) * 7.0
    o = oracle.readout(S, q, eps=0.0, scale=0.5)
    np.testing.assert_allclose(o, 0.5 * S @ (q / np.linalg.norm(q)), rtol=RTOL)


@pytest.mark.parametrize("V,K", [(1, 1), (3, 5), (8, 8), (7, 4)])
def test_step_equals_dense_gdn_formula(V, K):
    """S_t = exp(g) S_{t-1} (I - b k k^T) + b v k^T with dense matrices."""
    rng = np.random.default_rng(V * 100 + K)
    for trial in range(20):
        S = rng.normal(size=(V, K))
        v = rng.normal(size=V)
        k = rng.normal(size=K) * rng.uniform(0.2, 3.0)
        g = -rng.uniform(0, 5)
        beta = rng.uniform(0, 1)
        kh = _khat(k)
        dense = math.exp(g) * S @ (np.eye(K) - beta * np.outer(kh, kh)) + beta * np.outer(v, kh)
        got = oracle.step(S, v, k, g, beta)
        np.testing.assert_allclose(got, dense, rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("V,K", [(3, 5), (8, 8)])
def test_step_equals_dense_kda_formula(V, K):
    """KDA: S_t = S_{t-1} diag(exp(g)) (I - b k k^T) + b v k^T, g per key channel."""
    rng = np.random.default_rng(V * 7 + K)
    for trial in range(20):
        S = rng.normal(size=(V, K))
        v = rng.normal(size=V)
        k = rng.normal(size=K)
        g = -rng.uniform(0, 4, size=K)
        beta = rng.uniform(0, 1)
        kh = _khat(k)
        dense = S @ np.diag(np.exp(g)) @ (np.eye(K) - beta * np.outer(kh, kh)) \
            + beta * np.outer(v, kh)
        got = oracle.step(S, v, k, g, beta, per_key_gate=True)
        np.testing.assert_allclose(got, dense, rtol=1e-12, atol=1e-13)


def test_step_invariants():
    rng = np.random.default_rng(11)
    V, K = 6, 9
    S = rng.normal(size=(V, K))
    v = rng.normal(size=V)
    k = rng.normal(size=K)
    # beta = 0: pure decay
    np.testing.assert_allclose(oracle.step(S, v, k, -0.7, 0.0), math.exp(-0.7) * S, rtol=1e-15)
    # g = 0, beta = 0: identity, bit for bit
    assert np.array_equal(oracle.step(S, v, k, 0.0, 0.0), S)
    # beta = 1, |k^| = 1 (eps = 0): the delta rule overwrites, S_t k^ = v
    kh = _unit(k)
    S1 = oracle.step(S, v, kh, -0.3, 1.0, eps=0.0)
    np.testing.assert_allclose(S1 @ kh, v, rtol=0, atol=1e-13)
    # g -> -inf: the old state is gone, S_t = beta v k^T
    S2 = oracle.step(S, v, kh, -1e4, 0.37, eps=0.0)
    np.testing.assert_allclose(S2, 0.37 * np.outer(v, kh), rtol=1e-15, atol=0)


# ---------------------------------------------------------------- verify setup

def _random_layer(rng, d: oracle.Dims, io=gen.FP32):
    """A layer with random checkpoint and a garbage-filled ring (fp64 values of
    storage-rounded draws), plus window inputs."""
    ring = gen.garbage_ring(rng, d.num_slots, d.H, d.HV, d.L, d.K, d.V, io, d.per_key_gate)
    ly = oracle.Layer(d, checkpoint=rng.normal(size=(d.num_slots, d.HV, d.V, d.K)) * 0.5,
                      rawv=gen.to_f64(ring["rawv"]), rawk=gen.to_f64(ring["rawk"]),
                      ring_g=-np.abs(ring["g"].astype(np.float64)) * 2.0,
                      ring_beta=1.0 / (1.0 + np.exp(-ring["beta"].astype(np.float64))))
    return ly


def _window(rng, d: oracle.Dims, B, io=gen.FP32):
    w = gen.window_inputs(rng, B, d.T, d.H, d.HV, d.K, d.V, io, d.per_key_gate)
    A_log, dt_bias = gen.layer_params(rng, d.HV, d.K, d.per_key_gate)
    return {n: gen.to_f64(x) for n, x in w.items()}, A_log.astype(np.float64), \
        dt_bias.astype(np.float64)


def _ut_closed_form(d, S0, hist, win_k, win_v, win_q, win_g, win_beta, with_d=False):
    """Closed-form chunked UT transform of one (row, v-head) unit.

    Tokens 0..n-1 = W history records then T window tokens.  With per-token
    decay alpha_t = exp(g_t) and Gamma[i, r] = prod_{t=r+1..i} alpha_t:
        A[i, r] = beta_i Gamma[i, r] <k^_i, k^_r>            (r < i)
        R_i     = beta_i (v_i - Gamma[i, -1] S0 k^_i)
        D       = (I + A)^{-1} R          (rows d_i: the corrected deltas)
        o_s     = Gamma[s, -1] S0 q^_s + sum_{r <= s} Gamma[s, r] <k^_r, q^_s> d_r
    For KDA the decays are per key channel and sit inside the inner products.
    Returns outputs [T, V] computed with an explicit inverse (numpy) and with
    the exact finite Neumann sum of the nilpotent A; with_d: also D by both.
    """
    ks = [*hist["k"], *win_k]
    vs = [*hist["v"], *win_v]
    gs = [*hist["g"], *win_g]
    bs = [*hist["beta"], *win_beta]
    n = len(ks)
    W = n - d.T
    K = d.K
    kh = np.array([_khat(np.asarray(k)) for k in ks])
    qh = np.array([_khat(np.asarray(q)) for q in win_q])
    logal = np.array([np.broadcast_to(np.asarray(g, float), (K,)) for g in gs])  # [n, K]
    cum = np.concatenate([np.zeros((1, K)), np.cumsum(logal, axis=0)])  # cum[i+1] = sum_{t<=i}

    def decay(i, r):  # prod_{t=r+1..i} alpha_t as a [K] vector (r = -1: from the checkpoint)
        return np.exp(cum[i + 1] - cum[r + 1])

    A = np.zeros((n, n))
    R = np.zeros((n, d.V))
    for i in range(n):
        for r in range(i):
            A[i, r] = bs[i] * np.sum(kh[i] * kh[r] * decay(i, r))
        R[i] = bs[i] * (np.asarray(vs[i]) - S0 @ (decay(i, -1) * kh[i]))
    I = np.eye(n)
    D_inv = np.linalg.inv(I + A) @ R
    neu = sum(np.linalg.matrix_power(-A, p) for p in range(n))
    D_neu = neu @ R
    outs = []
    for D in (D_inv, D_neu):
        O = np.zeros((d.T, d.V))
        for s in range(d.T):
            i = W + s
            o = S0 @ (decay(i, -1) * qh[s])
            for r in range(i + 1):
                o = o + np.sum(kh[r] * qh[s] * decay(i, r)) * D[r]
            O[s] = d.scale * o
        outs.append(O)
    if with_d:
        return outs, (D_inv, D_neu)
    return outs


@pytest.mark.parametrize("per_key", [False, True])
@pytest.mark.parametrize("W", [0, 1, 5])
def test_verify_equals_closed_form_ut_transform(per_key, W):
    d = oracle.Dims(H=2, HV=4, K=6, V=5, T=4, L=16, num_slots=3, per_key_gate=per_key,
                    scale=0.75)
    rng = np.random.default_rng(100 + W + 10 * per_key)
    ly = _random_layer(rng, d)
    # mild decays so that every pair of tokens interacts
    ly.ring_g *= 0.05
    B = 2
    slot_idx = np.array([2, 0], np.int32)
    cur = oracle.Cursors(d.num_slots, write_pos=[W, 0, W], cache_base=[0, 0, 13])
    win, A_log, dt = _window(rng, d, B)
    win["a"] = win["a"] - 3.0  # weaker decay in the window too
    out, st = oracle.verify(d, ly.copy(), cur, slot_idx, win["q"], win["k"], win["v"], win["a"],
                            win["b"], A_log, dt)
    assert st == 0
    G = d.HV // d.H
    g_win, b_win = oracle.gate(A_log, win["a"], dt, win["b"], per_key_gate=per_key)
    for bb, slot in enumerate(slot_idx):
        base, wp = cur.cache_base[slot], cur.write_pos[slot]
        for hv in range(d.HV):
            h = hv // G
            pos = [(base + o) % d.L for o in range(wp)]
            hist = {"k": [ly.rawk[slot, h, p] for p in pos], "v": [ly.rawv[slot, hv, p] for p in pos],
                    "g": [ly.ring_g[slot, hv, p] for p in pos],
                    "beta": [ly.ring_beta[slot, hv, p] for p in pos]}
            o_inv, o_neu = _ut_closed_form(
                d, ly.checkpoint[slot, hv], hist, win["k"][bb, :, h], win["v"][bb, :, hv],
                win["q"][bb, :, h], list(g_win[bb, :, hv]), list(b_win[bb, :, hv]))
            np.testing.assert_allclose(out[bb, :, hv], o_inv, rtol=1e-9, atol=1e-11)
            np.testing.assert_allclose(out[bb, :, hv], o_neu, rtol=1e-9, atol=1e-11)


def test_verify_one_token_from_zero_state():
    """S0 = 0, W = 0, one window token: o = beta <k^, q^> v (scale 1)."""
    d = oracle.Dims(H=1, HV=1, K=8, V=3, T=1, L=2, num_slots=1)
    rng = np.random.default_rng(7)
    ly = oracle.Layer(d)
    q, k = rng.normal(size=(1, 1, 1, 8)), rng.normal(size=(1, 1, 1, 8))
    v = rng.normal(size=(1, 1, 1, 3))
    a, b = np.full((1, 1, 1), 0.4), np.full((1, 1, 1), -0.8)
    out, st = oracle.verify(d, ly, oracle.Cursors(1), [0], q, k, v, a, b, [0.5], [0.1])
    beta = 1 / (1 + math.exp(0.8))
    want = beta * float(_khat(k[0, 0, 0]) @ _khat(q[0, 0, 0])) * v[0, 0, 0]
    np.testing.assert_allclose(out[0, 0, 0], want, rtol=1e-13)


def test_verify_linear_in_state_and_values():
    d = oracle.Dims(H=2, HV=2, K=5, V=4, T=3, L=8, num_slots=1)
    rng = np.random.default_rng(8)
    ly1, ly2 = _random_layer(rng, d), _random_layer(rng, d)
    # same keys, gates and betas in both layers; only checkpoint and values differ
    ly2.rawk[:] = ly1.rawk
    ly2.ring_g[:] = ly1.ring_g
    ly2.ring_beta[:] = ly1.ring_beta
    win, A_log, dt = _window(rng, d, 1)
    v2 = rng.normal(size=win["v"].shape)
    cur = oracle.Cursors(1, write_pos=[3], cache_base=[6])
    c1, c2 = 0.7, -1.3
    ly3 = ly1.copy()
    ly3.checkpoint = c1 * ly1.checkpoint + c2 * ly2.checkpoint
    ly3.rawv = c1 * ly1.rawv + c2 * ly2.rawv
    o1, _ = oracle.verify(d, ly1.copy(), cur, [0], win["q"], win["k"], win["v"], win["a"],
                          win["b"], A_log, dt)
    o2, _ = oracle.verify(d, ly2.copy(), cur, [0], win["q"], win["k"], v2, win["a"], win["b"],
                          A_log, dt)
    o3, _ = oracle.verify(d, ly3, cur, [0], win["q"], win["k"], c1 * win["v"] + c2 * v2,
                          win["a"], win["b"], A_log, dt)
    np.testing.assert_allclose(o3, c1 * o1 + c2 * o2, rtol=1e-11, atol=1e-12)


def test_verify_touches_only_window_ring_slots_and_nothing_else():
    """Rejected drafts cost nothing: verify leaves the checkpoint and cursors
    bitwise untouched and writes exactly the ring positions (base + wp + s) & (L-1)."""
    d = oracle.Dims(H=2, HV=4, K=4, V=3, T=3, L=8, num_slots=4)
    rng = np.random.default_rng(9)
    ly = _random_layer(rng, d)
    before = ly.copy()
    cur = oracle.Cursors(4, write_pos=[2, 0, 5, 1], cache_base=[7, 0, 4, 3])
    cur0 = cur.copy()
    slot_idx = np.array([2, -1, 0], np.int32)
    win, A_log, dt = _window(rng, d, 3)
    out, st = oracle.verify(d, ly, cur, slot_idx, win["q"], win["k"], win["v"], win["a"],
                            win["b"], A_log, dt)
    assert st == 0
    assert np.array_equal(ly.checkpoint, before.checkpoint)
    for name in ("write_pos", "cache_base", "is_flush"):
        assert np.array_equal(getattr(cur, name), getattr(cur0, name))
    assert not out[1].any()  # padding row gives zeros
    written = set()
    for bb, slot in enumerate(slot_idx):
        if slot < 0:
            continue
        for s in range(d.T):
            written.add((slot, (cur.cache_base[slot] + cur.write_pos[slot] + s) % d.L))
    for slot in range(d.num_slots):
        for p in range(d.L):
            same = (np.array_equal(ly.rawv[slot, :, p], before.rawv[slot, :, p])
                    and np.array_equal(ly.rawk[slot, :, p], before.rawk[slot, :, p])
                    and np.array_equal(ly.ring_g[slot, :, p], before.ring_g[slot, :, p])
                    and np.array_equal(ly.ring_beta[slot, :, p], before.ring_beta[slot, :, p]))
            assert same == ((slot, p) not in written), (slot, p)
    # the written records are the raw window inputs
    for bb, slot in enumerate(slot_idx):
        if slot < 0:
            continue
        for s in range(d.T):
            p = (cur.cache_base[slot] + cur.write_pos[slot] + s) % d.L
            assert np.array_equal(ly.rawv[slot, :, p], win["v"][bb, s])
            assert np.array_equal(ly.rawk[slot, :, p], win["k"][bb, s])


def test_verify_status_and_padding_rows():
    d = oracle.Dims(H=1, HV=2, K=4, V=3, T=2, L=4, num_slots=2)
    rng = np.random.default_rng(10)
    ly = _random_layer(rng, d)
    win, A_log, dt = _window(rng, d, 3)
    cur = oracle.Cursors(2, write_pos=[3, 0], cache_base=[0, 0])
    out, st = oracle.verify(d, ly, cur, [0, 5, 1], win["q"], win["k"], win["v"], win["a"],
                            win["b"], A_log, dt)
    assert st == oracle.ST_RING_OVERFLOW | oracle.ST_SLOT_OOR
    assert not out[0].any() and not out[1].any() and out[2].any()


# ------------------------------------------------------- equivalences over rounds

def _run_protocol(d, rng, rounds, nslots=2):
    """Drive verify -> commit -> fold rounds in the oracle, keeping the true
    committed token list per (slot, v-head) on the side."""
    ly = _random_layer(rng, d)
    cur = oracle.Cursors(nslots)
    slot_idx = np.arange(nslots, dtype=np.int32)
    G = d.HV // d.H
    S_true = ly.checkpoint.copy()
    outs = []
    for r in range(rounds):
        win, A_log, dt = _window(rng, d, nslots)
        if r == 0:
            A0, dt0 = A_log, dt
        out, st = oracle.verify(d, ly, cur, slot_idx, win["q"], win["k"], win["v"], win["a"],
                                win["b"], A0, dt0)
        assert st == 0
        # the running committed state sees the window tokens directly
        g_win, b_win = oracle.gate(A0, win["a"], dt0, win["b"], per_key_gate=d.per_key_gate)
        acc = gen.accept_lens(rng, nslots, d.T)
        for bb in range(nslots):
            for hv in range(d.HV):
                S = S_true[bb, hv]
                for s in range(d.T):
                    S_run = oracle.step(S, win["v"][bb, s, hv], win["k"][bb, s, hv // G],
                                        g_win[bb, s, hv], b_win[bb, s, hv],
                                        per_key_gate=d.per_key_gate)
                    # output of a verify equals the readout of the running state
                    np.testing.assert_allclose(out[bb, s, hv],
                                               oracle.readout(S_run, win["q"][bb, s, hv // G],
                                                              scale=d.scale),
                                               rtol=1e-10, atol=1e-12)
                    if s < acc[bb]:
                        S_true[bb, hv] = S_run
                    S = S_run
        assert oracle.commit(d, cur, slot_idx, acc) == 0
        assert oracle.fold(d, ly, cur, slot_idx) == 0
        outs.append(out)
    return ly, cur, S_true


@pytest.mark.parametrize("per_key", [False, True])
def test_checkpoint_plus_ring_equals_running_state(per_key):
    d = oracle.Dims(H=1, HV=2, K=5, V=4, T=3, L=8, num_slots=2, per_key_gate=per_key)
    ly, cur, S_true = _run_protocol(d, np.random.default_rng(12 + per_key), rounds=9)
    # the checkpoint plus the unfolded history equals the running state
    dd = oracle.Dims(**{**d.__dict__})
    G = d.HV // d.H
    for slot in range(2):
        for hv in range(d.HV):
            pos = [(cur.cache_base[slot] + o) % d.L for o in range(cur.write_pos[slot])]
            S = oracle.run(dd, ly.checkpoint[slot, hv],
                           np.array([ly.rawv[slot, hv, p] for p in pos]).reshape(-1, d.V),
                           np.array([ly.rawk[slot, hv // G, p] for p in pos]).reshape(-1, d.K),
                           np.array([ly.ring_g[slot, hv, p] for p in pos]).reshape(len(pos), d.gw),
                           np.array([ly.ring_beta[slot, hv, p] for p in pos]))
            np.testing.assert_allclose(S, S_true[slot, hv], rtol=1e-11, atol=1e-12)


def test_fold_then_verify_equals_verify_with_history_bitwise():
    d = oracle.Dims(H=2, HV=4, K=6, V=5, T=4, L=16, num_slots=2)
    rng = np.random.default_rng(13)
    ly = _random_layer(rng, d)
    cur = oracle.Cursors(2, write_pos=[7, 3], cache_base=[12, 5], is_flush=[1, 1])
    win, A_log, dt = _window(rng, d, 2)
    args = (win["q"], win["k"], win["v"], win["a"], win["b"], A_log, dt)
    o_hist, _ = oracle.verify(d, ly.copy(), cur.copy(), [0, 1], *args)
    ly2, cur2 = ly.copy(), cur.copy()
    assert oracle.fold(d, ly2, cur2, [0, 1]) == 0
    assert list(cur2.write_pos) == [0, 0] and list(cur2.is_flush) == [0, 0]
    assert list(cur2.cache_base) == [(12 + 7) % 16, (5 + 3) % 16]
    o_fold, _ = oracle.verify(d, ly2, cur2, [0, 1], *args)
    assert np.array_equal(o_hist, o_fold)


def test_fold_skips_rows_without_flag_and_is_idempotent():
    d = oracle.Dims(H=1, HV=1, K=4, V=3, T=2, L=8, num_slots=3)
    rng = np.random.default_rng(14)
    ly = _random_layer(rng, d)
    cur = oracle.Cursors(3, write_pos=[5, 5, 2], cache_base=[1, 2, 3], is_flush=[1, 0, 1])
    before = ly.copy()
    assert oracle.fold(d, ly, cur, [0, 1, -1]) == 0
    assert not np.array_equal(ly.checkpoint[0], before.checkpoint[0])
    assert np.array_equal(ly.checkpoint[1:], before.checkpoint[1:])
    assert list(cur.write_pos) == [0, 5, 2] and list(cur.cache_base) == [6, 2, 3]
    snap = ly.copy()
    assert oracle.fold(d, ly, cur, [0, 1]) == 0  # nothing flagged any more
    assert np.array_equal(ly.checkpoint, snap.checkpoint)


def test_commit_status_bits():
    d = oracle.Dims(H=1, HV=1, K=2, V=2, T=4, L=16, num_slots=2)
    cur = oracle.Cursors(2)
    st = oracle.commit(d, cur, [0, 1, 7, -1], [5, 2, 1, 3])
    assert st == oracle.ST_ACCEPT_RANGE | oracle.ST_SLOT_OOR
    assert list(cur.write_pos) == [0, 2]
    st = oracle.commit(d, cur, [0], [-1])
    assert st == oracle.ST_ACCEPT_RANGE


def test_commit_skips_rows_with_corrupt_cursors():
    """A row whose cursors are outside the ring (write_pos outside [0, L] or
    cache_base outside [0, L), the rule verify applies) is left exactly as it is
    and reported; the other rows commit normally."""
    d = oracle.Dims(H=1, HV=1, K=2, V=2, T=4, L=16, num_slots=5)
    cur = oracle.Cursors(5, write_pos=[-1, 17, 3, 16, 2], cache_base=[0, 0, 16, 15, -2],
                         is_flush=[0, 0, 0, 1, 0])
    before = cur.copy()
    st = oracle.commit(d, cur, [0, 1, 2, 3, 4], [1, 1, 1, 0, 1])
    assert st == oracle.ST_CURSOR_CORRUPT
    for name in ("write_pos", "cache_base", "is_flush"):
        got, want = getattr(cur, name), getattr(before, name)
        assert list(got[[0, 1, 2, 4]]) == list(want[[0, 1, 2, 4]]), name
    # the edge write_pos == L is in range: it commits (accept 0) and stays flagged
    assert cur.write_pos[3] == 16 and cur.is_flush[3] == 1
