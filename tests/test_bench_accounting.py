"""The benchmark's byte accounting and cursor mirror, on the CPU.

The roofline fraction divides algorithmic bytes by time, so the byte formula
is pinned here to the per-term sum written out (checkpoint, history records,
window inputs, outputs, ring write) at the Qwen3-Next shape, and the host
mirror of the cursors (which gives each verify's ring fill W) is pinned to the
oracle's commit and fold."""
import numpy as np

import bench
import oracle
from gated_delta_rule_spec_gb300 import inputs as gen


def test_verify_bytes_at_the_qwen3next_shape():
    K = V = 128
    T, G, e = 4, 2, 2
    for W in (0, 1, 29, 60):
        per_term = (V * K * 4                              # checkpoint tile
                    + W * (V * e + K * e // G + 4 + 4)     # history: raw v, raw k share, g, beta
                    + T * (2 * K * e // G + V * e + 2 * e)  # window q, k shares, v, a, b
                    + T * V * e                             # outputs
                    + T * (V * e + K * e // G + 4 + 4))    # ring write of the window
        got = float(bench.verify_bytes_per_unit(np.array(W), K, V, T, G, e, False))
        assert got == per_term == 70192 + 392 * W


def test_kda_bytes_scale_the_gate_terms_by_k():
    K = V = 128
    T, G, e = 4, 2, 2
    W = 10
    gdn = float(bench.verify_bytes_per_unit(np.array(W), K, V, T, G, e, False))
    kda = float(bench.verify_bytes_per_unit(np.array(W), K, V, T, G, e, True))
    # per record and per window token the gate grows from one value to K
    assert kda - gdn == W * 4 * (K - 1) + T * e * (K - 1) + T * 4 * (K - 1)


def test_snapshot_bytes():
    K = V = 128
    T, G, e = 4, 2, 2
    state = V * K * 4
    assert bench.snapshot_bytes_per_unit(K, V, T, G, e) == \
        state + T * state + T * (2 * K * e / G + V * e + 2 * e) + T * V * e + 2 * state


def test_cursor_mirror_matches_the_oracle_protocol():
    T, L, B = 4, 64, 32
    rng = np.random.default_rng(3)
    d = oracle.Dims(H=1, HV=1, K=4, V=4, T=T, L=L, num_slots=B)
    wp0 = rng.integers(0, L - 2 * T + 1, B).astype(np.int32)
    cur = oracle.Cursors(B, wp0.copy(), rng.integers(0, L, B).astype(np.int32), np.zeros(B, np.int32))
    ly = oracle.Layer(d)
    slots = np.arange(B, dtype=np.int32)
    accs = [gen.accept_lens(rng, B, T) for _ in range(120)]
    W = bench.mirror_cursors(wp0, None, accs, T, L)
    for step, acc in enumerate(accs):
        assert np.array_equal(W[step], cur.write_pos), step
        assert oracle.commit(d, cur, slots, acc) == 0
        assert oracle.fold(d, ly, cur, slots) == 0


def test_chunk_prefill_flops():
    """One full 64-token chunk and a one-token tail, term by term: the Gram of
    keys and queries against the keys, the state products of keys and queries,
    the intra-chunk outputs, the state update."""
    wl = bench.Workload(1)
    K, V = wl.K, wl.V

    def chunk(n):
        return 2 * K * (2 * n) * n + 2 * V * K * (2 * n) + 2 * V * n * n + 2 * V * K * n

    assert bench._prefill_chunk_flops(1, 65, wl) == (chunk(64) + chunk(1)) * wl.HV
    assert bench._prefill_chunk_flops(3, 128, wl) == 3 * 2 * chunk(64) * wl.HV
    assert bench._prefill_chunk_flops(2, 0, wl) == 0
