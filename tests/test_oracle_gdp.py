"""Pins for the stacked-Householder (Gated DeltaProduct-style) oracle, CPU only.

Per token the gate once, then n_h delta-rule steps with their own (k, v, beta). Pins that share no code with it:
- n_h = 1 is the Gated DeltaNet update (the GDN oracle);
- a second step with beta = 0 changes nothing (n_h = 2 reduces to GDN);
- the token's transition on the state is the explicit matrix e^g (I - b_n k_n k_n^T) ... (I - b_1 k_1 k_1^T), and its
  write term sum_h (prod_{h' > h} (I - b_h' k_h' k_h'^T)) b_h k_h v_h^T, formed as dk x dk matrices in NumPy;
- with the write terms only on one step, the generic DPLR oracle with the explicit A, B (rank n_h) gives the same
  outputs (the product of n_h Householders is identity minus a rank-n_h term).
"""

import numpy as np

import oracle


def _inputs(seed, nh, H=1, T=6, dk=4, dv=3):
    rng = np.random.default_rng(seed)
    k = rng.standard_normal((1, H, T, nh, dk))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    return dict(q=rng.standard_normal((1, H, T, dk)), k=k, v=rng.standard_normal((1, H, T, nh, dv)),
                g=-np.abs(rng.standard_normal((1, H, T))) * 0.3, beta=rng.uniform(0.1, 1.9, (1, H, T, nh)),
                S0=0.3 * rng.standard_normal((1, H, dk, dv)))


def test_one_step_is_gated_deltanet():
    a = _inputs(1, 1)
    o, ST = oracle.gdp(**a)
    o2, ST2 = oracle.forward("gdn", a["q"], a["k"][:, :, :, 0], a["v"][:, :, :, 0], a["g"], a["beta"][..., 0], S0=a["S0"])
    assert np.allclose(o, o2, atol=1e-13) and np.allclose(ST, ST2, atol=1e-13)


def test_second_step_with_zero_beta_is_gated_deltanet():
    a = _inputs(2, 2)
    a["beta"][..., 1] = 0.0
    o, ST = oracle.gdp(**a)
    o2, ST2 = oracle.forward("gdn", a["q"], a["k"][:, :, :, 0], a["v"][:, :, :, 0], a["g"], a["beta"][..., 0], S0=a["S0"])
    assert np.allclose(o, o2, atol=1e-13) and np.allclose(ST, ST2, atol=1e-13)


def _explicit(a, nh):
    """The recurrence with each token's transition and write formed as explicit dk x dk / dk x dv matrices."""
    q, k, v, g, beta = (a[x][0, 0] for x in ("q", "k", "v", "g", "beta"))
    T, dk = q.shape
    S = a["S0"][0, 0].copy()
    outs = []
    for t in range(T):
        H = [np.eye(dk) - beta[t, h] * np.outer(k[t, h], k[t, h]) for h in range(nh)]
        P = np.eye(dk)
        for h in range(nh):
            P = H[h] @ P
        W = np.zeros((dk, v.shape[-1]))
        for h in range(nh):
            M = np.eye(dk)
            for h2 in range(h + 1, nh):
                M = H[h2] @ M
            W += M @ np.outer(beta[t, h] * k[t, h], v[t, h])
        S = np.exp(g[t]) * (P @ S) + W
        outs.append(S.T @ q[t])
    return np.array(outs), S


def test_explicit_transition_and_write():
    for nh in (2, 3):
        a = _inputs(3 + nh, nh)
        o, ST = oracle.gdp(**a)
        o2, ST2 = _explicit(a, nh)
        assert np.allclose(o[0, 0], o2, atol=1e-12) and np.allclose(ST[0, 0], ST2, atol=1e-12)


def test_rank_nh_transition_in_the_generic_form():
    """The transition is e^g (I - A B^T) with A = [k_1 .. k_n] and B columns b_h = beta_h (k_h - sum_{h'<h} (k_h'.k_h) b_h'):
    the generic oracle with those factors (writes off) matches."""
    nh = 3
    a = _inputs(9, nh)
    a["v"] = np.zeros_like(a["v"])
    o, ST = oracle.gdp(**a)
    k, beta, g = a["k"][0, 0], a["beta"][0, 0], a["g"][0, 0]
    T, dk = a["q"].shape[2], a["q"].shape[3]
    A = np.zeros((1, 1, T, nh, dk))
    Bm = np.zeros((1, 1, T, nh, dk))
    for t in range(T):
        bs = []
        for h in range(nh):
            b = k[t, h].copy()
            for h2 in range(h):
                b -= (k[t, h2] @ k[t, h]) * bs[h2]
            b *= beta[t, h]
            bs.append(b)
            A[0, 0, t, h] = np.exp(g[t]) * k[t, h]
            Bm[0, 0, t, h] = b
    decay = np.repeat(g[None, None, :, None], dk, axis=3)
    o2, ST2 = oracle.forward("generic", a["q"], decay=decay, A=A, Bm=Bm, K=np.zeros((1, 1, T, 0, dk)),
                             V=np.zeros((1, 1, T, 0, 3)), S0=a["S0"])
    assert np.allclose(o, o2, atol=1e-12) and np.allclose(ST, ST2, atol=1e-12)
