"""Pins of the cursor arithmetic (commit, fold, reset) and ring indexing.

The pages' own protocol ("A", the blog post on PR #28695, §4.4, §8.1 and
§9.3) folds inside the next verify and moves the cursors in commit:
    if is_flush: cache_base = (cache_base + write_pos) & (L-1); write_pos = acc
    else:        write_pos += acc
    is_flush = (write_pos + 2T > L)
The library calls the fold as its own step between commit and the next verify
(protocol "B"): commit does write_pos += acc and sets is_flush the same way;
fold moves cache_base by write_pos and clears write_pos and is_flush.

The tests show by exhaustive simulation that both protocols put every record
at the same ring position and fold the same records at the same point of the
token stream, that a verify never runs past the ring (write_pos + T <= L) and
that the oracle's commit/fold/reset follow protocol B; and they check the
cursor examples printed on the pages (tests/golden/cursor_examples.json).
"""
import itertools
import json
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "cursor_examples.json")


def _protocol_a(L, T, accs):
    base = wp = flag = 0
    committed = 0
    pos = {}
    rounds = []
    for acc in accs:
        assert wp + T <= L, "verify would run past the ring"
        hist = list(range(committed - wp, committed))
        for o, gidx in enumerate(hist):
            assert pos[gidx] == (base + o) & (L - 1)
        window = [(base + wp + s) & (L - 1) for s in range(T)]
        folded_here = hist if flag else []
        for s in range(acc):
            pos[committed + s] = window[s]
        committed += acc
        if flag:
            base = (base + wp) & (L - 1)
            wp = acc
        else:
            wp += acc
        flag = int(wp + 2 * T > L)
        rounds.append({"window": window, "hist": hist, "folded_at_verify": folded_here})
    return pos, rounds


def _protocol_b(L, T, accs):
    base = wp = flag = 0
    committed = 0
    pos = {}
    rounds = []
    states = []
    for acc in accs:
        assert wp + T <= L, "verify would run past the ring"
        assert flag == 0
        hist = list(range(committed - wp, committed))
        for o, gidx in enumerate(hist):
            assert pos[gidx] == (base + o) & (L - 1)
        window = [(base + wp + s) & (L - 1) for s in range(T)]
        for s in range(acc):
            pos[committed + s] = window[s]
        committed += acc
        wp += acc                                  # commit
        flag = int(wp + 2 * T > L)
        folded_after = list(range(committed - wp, committed)) if flag else []
        if flag:                                   # fold
            base = (base + wp) & (L - 1)
            wp = 0
            flag = 0
        rounds.append({"window": window, "hist": hist, "folded_after_commit": folded_after})
        states.append((base, wp, flag))
    return pos, rounds, states


def _check_equivalent(L, T, accs):
    pos_a, ra = _protocol_a(L, T, accs)
    pos_b, rb, _ = _protocol_b(L, T, accs)
    assert pos_a == pos_b
    for i, (a, b) in enumerate(zip(ra, rb)):
        assert a["window"] == b["window"], (L, T, accs, i)
        if a["folded_at_verify"]:
            # A folds at verify i exactly what B folded after commit i-1
            assert a["folded_at_verify"] == rb[i - 1]["folded_after_commit"]
            assert b["hist"] == []
        else:
            assert a["hist"] == b["hist"]


@pytest.mark.parametrize("L,T", [(8, 1), (8, 2), (8, 3), (8, 4), (16, 1), (16, 2), (16, 3),
                                 (16, 4), (64, 1), (64, 4)])
def test_protocols_a_and_b_agree_exhaustively(L, T):
    depth = 6
    for accs in itertools.product(range(T + 1), repeat=depth):
        _check_equivalent(L, T, accs)


@pytest.mark.parametrize("L,T", [(16, 4), (64, 4), (64, 8), (128, 4)])
def test_protocols_agree_on_long_random_runs(L, T):
    rng = np.random.default_rng(L * 31 + T)
    for _ in range(300):
        accs = rng.integers(0, T + 1, size=200).tolist()
        _check_equivalent(L, T, accs)


def _oracle_dims(L, T, n):
    return oracle.Dims(H=1, HV=1, K=1, V=1, T=T, L=L, num_slots=n)


@pytest.mark.parametrize("L,T", [(8, 4), (16, 4), (64, 4), (8, 2)])
def test_oracle_cursors_follow_protocol_b(L, T):
    rng = np.random.default_rng(L + 7 * T)
    nslots = 5
    d = _oracle_dims(L, T, nslots)
    ly = oracle.Layer(d)
    cur = oracle.Cursors(nslots)
    slot_idx = np.arange(nslots, dtype=np.int32)
    seqs = rng.integers(0, T + 1, size=(nslots, 150))
    expect = [_protocol_b(L, T, seqs[i].tolist())[2] for i in range(nslots)]
    for r in range(seqs.shape[1]):
        assert oracle.commit(d, cur, slot_idx, seqs[:, r]) == 0
        assert oracle.fold(d, ly, cur, slot_idx) == 0
        for i in range(nslots):
            assert (cur.cache_base[i], cur.write_pos[i], cur.is_flush[i]) == expect[i][r]


def test_golden_accept_walk():
    ex = json.load(open(GOLDEN))["accept_walk"]
    L, T = 256, ex["drafts"]
    d = _oracle_dims(L, T, 1)
    cur = oracle.Cursors(1, write_pos=[ex["write_pos_before"]])
    offs = [(cur.cache_base[0] + cur.write_pos[0] + s) & (L - 1) for s in range(T)]
    assert offs == ex["draft_offsets"]
    assert oracle.commit(d, cur, [0], [ex["accept_len"]]) == 0
    assert cur.write_pos[0] == ex["write_pos_after"]


def test_golden_ring_walk_l8():
    ex = json.load(open(GOLDEN))["ring_walk_L8"]
    L = ex["L"]
    phys = [(ex["base_before"] + o) & (L - 1) for o in ex["logical_offsets"]]
    assert phys == ex["physical_slots"]
    d = _oracle_dims(L, 2, 1)
    cur = oracle.Cursors(1, write_pos=[ex["write_pos_before"]],
                         cache_base=[ex["base_before"]], is_flush=[1])
    assert oracle.fold(d, oracle.Layer(d), cur, [0]) == 0
    assert cur.cache_base[0] == ex["base_after_fold"] and cur.write_pos[0] == 0


def test_golden_margin_rule():
    for c in json.load(open(GOLDEN))["margin_rule"]["cases"]:
        d = _oracle_dims(c["L"], c["T"], 1)
        cur = oracle.Cursors(1)
        assert oracle.commit(d, cur, [0], [0]) == 0
        cur.write_pos[0] = c["write_pos"]
        assert oracle.commit(d, cur, [0], [0]) == 0
        assert cur.is_flush[0] == c["is_flush"], c


def test_reset_zeroes_only_named_slots():
    d = _oracle_dims(16, 4, 4)
    cur = oracle.Cursors(4, write_pos=[3, 4, 5, 6], cache_base=[1, 2, 3, 4], is_flush=[1, 0, 1, 0])
    assert oracle.reset(d, cur, [2, -1, 0]) == 0
    assert list(cur.write_pos) == [0, 4, 0, 6]
    assert list(cur.cache_base) == [0, 2, 0, 4]
    assert list(cur.is_flush) == [0, 0, 0, 0]
    assert oracle.reset(d, cur, [9]) == oracle.ST_SLOT_OOR
