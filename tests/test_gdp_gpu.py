"""Stacked Householders (dplr_gdp_forward, Gated DeltaProduct-style) against the float64 oracle (oracle.gdp).

Whole small problems, element by element: max |err| <= 1e-4 of the RMS for o and S_T (the factors are built in
fp32 from the exact inputs and the generic path keeps fp32-level accuracy). dk = dv = 64 with n_h <= 2 runs the
generic tensor-core path; the other shapes the fp32 two-stage path.
"""

import numpy as np
import pytest

import oracle

pytestmark = pytest.mark.gpu

TAU = 1e-4


@pytest.fixture(scope="module")
def sdl():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from structured_decay_linear_gb300 import build as nvbuild
    nvbuild.build()
    import structured_decay_linear_gb300 as s
    s.library()
    return s


def _rel(a, ref):
    return float(np.abs(a - ref).max() / max(np.sqrt(np.mean(ref ** 2)), 1e-30))


def _inputs(seed, H, T, dk, dv, nh, dtype):
    rng = np.random.default_rng(seed)
    k = rng.standard_normal((1, H, T, nh, dk)).astype(np.float32)
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    a = dict(q=(rng.standard_normal((1, H, T, dk)) / np.sqrt(dk)).astype(np.float32), k=k,
             v=rng.standard_normal((1, H, T, nh, dv)).astype(np.float32),
             g=(-np.logaddexp(0, -(rng.standard_normal((1, H, T)) + 3))).astype(np.float32),
             beta=(2 / (1 + np.exp(-rng.standard_normal((1, H, T, nh))))).astype(np.float32),
             S0=(0.1 * rng.standard_normal((1, H, dk, dv))).astype(np.float32))
    if dtype == "bf16":
        import workloads
        for x in ("q", "k", "v"):
            a[x] = workloads.round_to_bf16(a[x])
    return a


@pytest.mark.parametrize("dtype,dk,dv,nh,H,T,path", [
    ("f32", 64, 64, 2, 2, 200, "generic_tcgen05"),
    ("bf16", 64, 64, 1, 2, 97, "generic_tcgen05"),
    ("f32", 64, 64, 3, 1, 130, "two_stage_fp32"),
    ("bf16", 128, 128, 2, 2, 150, "two_stage_fp32"),
    ("f32", 32, 64, 3, 1, 40, "two_stage_fp32"),
])
def test_gdp_matches_oracle(sdl, dtype, dk, dv, nh, H, T, path):
    import torch
    a = _inputs(700 + nh + dk, H, T, dk, dv, nh, dtype)
    dt = torch.bfloat16 if dtype == "bf16" else torch.float32
    d = lambda x, t: torch.from_numpy(np.ascontiguousarray(x)).to("cuda").to(t)
    f = sdl.GDP(dt, 1, H, T, dk, dv, nh)
    assert f.path == path
    o, ST = f(d(a["q"], dt), d(a["k"], dt), d(a["v"], dt), d(a["g"], torch.float32), d(a["beta"], torch.float32),
              d(a["S0"], torch.float32))
    torch.cuda.synchronize()
    o_ref, S_ref = oracle.gdp(a["q"], a["k"], a["v"], a["g"], a["beta"], a["S0"])
    assert _rel(o.double().cpu().numpy(), o_ref) <= TAU
    assert _rel(ST.double().cpu().numpy(), S_ref) <= TAU
