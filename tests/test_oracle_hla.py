"""Pins for the HLA composition oracle (oracle.hla), CPU only.

HLA's query-conditioned state composes the exact chunk summaries (A_j, B_j) of the Gated DeltaNet updates with
per-query gates, S <- ((1 - w) I + w A_j) S + w B_j, then runs the current chunk's causal prefix ("HLA: Expressive
Hybrid Linear Attention via Chunk-Wise Dynamic Mixing", Method step 5). The pins use only the GDN forward oracle:
- every gate 1: the composition is the plain GDN recurrence (the summaries are exact, Prerequisites: affine closure);
- every gate 0: each chunk restarts from a zero state;
- one gate 1 and the rest 0: the history is chunk j alone, so the output is that of the GDN recurrence over chunk
  j's tokens followed by the current chunk's prefix;
- the threshold: gates below it act as zero;
- one gate at 0.5: the output is affine in each gate (the mean of the outputs at 0 and 1).
"""

import numpy as np

import oracle


def _inputs(seed, H=2, T=20, dk=4, dv=3):
    rng = np.random.default_rng(seed)
    k = rng.standard_normal((1, H, T, dk))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    return dict(q=rng.standard_normal((1, H, T, dk)), k=k, v=rng.standard_normal((1, H, T, dv)),
                g=-np.abs(rng.standard_normal((1, H, T))) * 0.2, beta=rng.uniform(0.1, 1.0, (1, H, T)))


def test_all_gates_one_is_the_gdn_recurrence():
    a = _inputs(1)
    T, L = 20, 6
    W = np.ones((1, 2, T, (T + L - 1) // L))
    o = oracle.hla(a["q"], a["k"], a["v"], a["g"], a["beta"], W, L)
    o_ref, _ = oracle.forward("gdn", a["q"], a["k"], a["v"], a["g"], a["beta"])
    assert np.allclose(o, o_ref, rtol=1e-12, atol=1e-12)


def test_all_gates_zero_restarts_each_chunk():
    a = _inputs(2)
    T, L = 20, 6
    W = np.zeros((1, 2, T, 4))
    o = oracle.hla(a["q"], a["k"], a["v"], a["g"], a["beta"], W, L)
    for c0 in range(0, T, L):
        sl = slice(c0, min(T, c0 + L))
        o_ref, _ = oracle.forward("gdn", *(a[x][:, :, sl] for x in ("q", "k", "v", "g", "beta")))
        assert np.allclose(o[:, :, sl], o_ref, rtol=1e-12, atol=1e-12)


def test_one_gate_selects_one_chunk_of_history():
    a = _inputs(3, H=1)
    T, L = 20, 5
    i, j = 17, 1                        # query in chunk 3, history chunk 1 only
    W = np.zeros((1, 1, T, 4))
    W[0, 0, i, j] = 1.0
    o = oracle.hla(a["q"], a["k"], a["v"], a["g"], a["beta"], W, L)
    toks = list(range(j * L, (j + 1) * L)) + list(range((i // L) * L, i + 1))
    sub = {x: a[x][:, :, toks] for x in ("q", "k", "v", "g", "beta")}
    o_ref, _ = oracle.forward("gdn", sub["q"], sub["k"], sub["v"], sub["g"], sub["beta"])
    assert np.allclose(o[0, 0, i], o_ref[0, 0, -1], rtol=1e-12, atol=1e-12)


def test_gates_below_the_threshold_are_zero():
    T, L = 18, 6
    a = _inputs(4, T=T)
    rng = np.random.default_rng(5)
    W = rng.uniform(0.0, 1.0, (1, 2, T, 3))
    Wz = np.where(W < 0.4, 0.0, W)
    o1 = oracle.hla(a["q"], a["k"], a["v"], a["g"], a["beta"], W, L, theta=0.4)
    o2 = oracle.hla(a["q"], a["k"], a["v"], a["g"], a["beta"], Wz, L)
    assert np.array_equal(o1, o2)


def test_output_is_affine_in_each_gate():
    T, L = 16, 4
    a = _inputs(6, H=1, T=T)
    rng = np.random.default_rng(7)
    W = rng.uniform(0.2, 1.0, (1, 1, T, 4))
    i, j = 14, 1
    outs = []
    for wv in (0.0, 0.5, 1.0):
        W2 = W.copy()
        W2[0, 0, i, j] = wv
        outs.append(oracle.hla(a["q"], a["k"], a["v"], a["g"], a["beta"], W2, L)[0, 0, i])
    assert np.allclose(outs[1], 0.5 * (outs[0] + outs[2]), rtol=1e-12, atol=1e-12)
    assert not np.allclose(outs[0], outs[2])
