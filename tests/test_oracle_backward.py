"""Pins for the oracle's reverse mode (oracle.backward), CPU only.

The backward oracle differentiates the serial recurrence token by token. It is pinned against things
that do not share its code:
- central finite differences of the forward oracle (float64, step 1e-6) for every input of every mode,
  on tiny problems where each derivative costs two forward calls;
- closed forms: with beta = 0 and D = I (causal linear attention, Log-Linear Attention page, Framework:
  O = (Q K^T masked) V plus the initial state's readout) the gradients of q, v and S0 are sums that can
  be written down directly; with the write term off, dS0 is the transposed product of the token maps
  applied to dS_T.
"""

import numpy as np
import pytest

import oracle

H_FD = 1e-6


def _loss(mode, args, do, dST):
    o, ST = oracle.forward(mode, **args)
    return float((o * do).sum() + (ST * dST).sum())


def _fd_check(mode, args, names, seed):
    rng = np.random.default_rng(seed)
    B, H, T, _ = args["q"].shape
    dv = args["v"].shape[3] if args.get("v") is not None else args["V"].shape[4]
    dk = args["q"].shape[3]
    do = rng.standard_normal((B, H, T, dv))
    dST = rng.standard_normal((B, H, dk, dv))
    g = oracle.backward(mode, do=do, dST=dST, **args)
    for name in names:
        x = args[name]
        fd = np.zeros_like(x)
        for idx in np.ndindex(*x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += H_FD
            xm[idx] -= H_FD
            fd[idx] = (_loss(mode, {**args, name: xp}, do, dST) - _loss(mode, {**args, name: xm}, do, dST)) / (2 * H_FD)
        err = np.abs(fd - g[name]).max()
        assert err <= 1e-6 * max(1.0, np.abs(fd).max()), f"{mode} d{name}: max |fd - backward| = {err:.3e}"


def _structured(seed, T=5, dk=4, dv=3, H=2, hdla=False):
    rng = np.random.default_rng(seed)
    k = rng.standard_normal((1, H, T, dk))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    decay = -np.abs(rng.standard_normal((1, H, T, dk) if hdla else (1, H, T))) * 0.3
    return dict(q=rng.standard_normal((1, H, T, dk)), k=k, v=rng.standard_normal((1, H, T, dv)), decay=decay,
                beta=rng.uniform(0.1, 1.8, (1, H, T)), S0=0.3 * rng.standard_normal((1, H, dk, dv)))


def _generic(seed, T=5, dk=4, dv=3, H=1, r=2, p=1):
    rng = np.random.default_rng(seed)
    return dict(q=rng.standard_normal((1, H, T, dk)), decay=-np.abs(rng.standard_normal((1, H, T, dk))) * 0.3,
                A=0.5 * rng.standard_normal((1, H, T, r, dk)), Bm=0.5 * rng.standard_normal((1, H, T, r, dk)),
                K=rng.standard_normal((1, H, T, p, dk)), V=rng.standard_normal((1, H, T, p, dv)),
                S0=0.3 * rng.standard_normal((1, H, dk, dv)))


def test_gdn_backward_matches_finite_differences():
    _fd_check("gdn", _structured(1), ["q", "k", "v", "decay", "beta", "S0"], seed=11)


def test_hdla_backward_matches_finite_differences():
    _fd_check("hdla", _structured(2, hdla=True), ["q", "k", "v", "decay", "beta", "S0"], seed=12)


@pytest.mark.parametrize("r,p", [(2, 1), (1, 0), (3, 2)])
def test_generic_backward_matches_finite_differences(r, p):
    args = _generic(3 + r, r=r, p=p)
    names = ["q", "decay", "A", "Bm", "S0"] + (["K", "V"] if p else [])
    if p == 0:   # no write term: a zero-rank K, V (V still fixes dv)
        args["K"] = np.zeros((1, 1, 5, 0, 4))
        args["V"] = np.zeros((1, 1, 5, 0, 3))
    _fd_check("generic", args, names, seed=13 + r)


def test_linear_attention_closed_form():
    """beta = 0, D = I: o_t = S0^T q_t + sum_{s<=t} (q_t . k_s) v_s, so dq_t = S0 do_t + sum_{s<=t} k_s (v_s . do_t),
    dv_s = sum_{t>=s} (q_t . k_s) do_t + dST^T k_s and dS0 = sum_t q_t do_t^T + dST, written out directly."""
    rng = np.random.default_rng(7)
    T, dk, dv = 7, 5, 4
    q, k, v = rng.standard_normal((T, dk)), rng.standard_normal((T, dk)), rng.standard_normal((T, dv))
    S0, do, dST = rng.standard_normal((dk, dv)), rng.standard_normal((T, dv)), rng.standard_normal((dk, dv))
    # generic mode: D = I (log-decay 0), no factors (A = B = 0), write K_t V_t^T = k_t v_t^T
    g = oracle.backward("generic", q[None, None], decay=np.zeros((1, 1, T, dk)), A=np.zeros((1, 1, T, 1, dk)),
                        Bm=np.zeros((1, 1, T, 1, dk)), K=k[None, None, :, None], V=v[None, None, :, None],
                        S0=S0[None, None], do=do[None, None], dST=dST[None, None])
    dq = np.array([S0 @ do[t] + sum(k[s] * (v[s] @ do[t]) for s in range(t + 1)) for t in range(T)])
    dvv = np.array([sum((q[t] @ k[s]) * do[t] for t in range(s, T)) + dST.T @ k[s] for s in range(T)])
    dS0 = sum(np.outer(q[t], do[t]) for t in range(T)) + dST
    assert np.allclose(g["q"][0, 0], dq, atol=1e-12)
    assert np.allclose(g["V"][0, 0, :, 0], dvv, atol=1e-12)
    assert np.allclose(g["S0"][0, 0], dS0, atol=1e-12)


def test_state_gradient_is_the_transposed_map():
    """With the write term off (beta = 0 in GDN) and do = 0, S_T = e^{sum g} S0, so dS0 = e^{sum g} dS_T."""
    rng = np.random.default_rng(8)
    T, dk, dv = 6, 3, 2
    a = _structured(9, T=T, dk=dk, dv=dv, H=1)
    a["beta"] = np.zeros_like(a["beta"])
    dST = rng.standard_normal((1, 1, dk, dv))
    g = oracle.backward("gdn", do=np.zeros((1, 1, T, dv)), dST=dST, **a)
    assert np.allclose(g["S0"], np.exp(a["decay"].sum()) * dST, atol=1e-13)
    assert np.allclose(g["q"], 0.0) and np.allclose(g["v"], 0.0)
