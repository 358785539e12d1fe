"""The backward (dplr_la_backward) against the float64 reverse-mode oracle (oracle.backward).

Every gradient the mode has is compared element by element over whole small problems that span several of the
backward's blocks and a ragged last one: max |err| <= TAU * RMS of the oracle's gradient. The backward computes in
fp32 from exact inputs (bf16 values upcast), through the WY factors of blocks of 16 to 32 tokens; TAU = 1e-3 allows
for the fp32 rounding of those block products (the measured errors sit near 1e-5).
"""

import numpy as np
import pytest

import oracle
import workloads

pytestmark = pytest.mark.gpu

TAU = 1e-3


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


def _run(sdl, mode, dtype, inp, do, dST):
    import torch
    dt = torch.bfloat16 if dtype == "bf16" else torch.float32
    d = lambda x, t: None if x is None else torch.from_numpy(np.ascontiguousarray(x)).to("cuda").to(t)
    B, H, T = inp["B"], inp["H"], inp["T"]
    dk = inp["q"].shape[3]
    dv = do.shape[3]
    r = inp["A"].shape[3] if inp["A"] is not None else None
    p = (inp["K"].shape[3] if inp["K"] is not None else 0) if mode == "generic" else None
    bw = sdl.Backward(mode, dt, B, H, T, dk, dv, r, p)
    g = bw(dO=d(do, torch.float32), dST=d(dST, torch.float32), q=d(inp["q"], dt), k=d(inp["k"], dt),
           v=d(inp["v"], dt), decay=d(inp["decay"], torch.float32), beta=d(inp["beta"], torch.float32),
           A=d(inp["A"], dt), Bm=d(inp["Bm"], dt), K=d(inp["K"], dt), V=d(inp["V"], dt),
           S0=d(inp["S0"], torch.float32))
    torch.cuda.synchronize()
    return {k2: v2.double().cpu().numpy() for k2, v2 in g.items()}


def _check(g, ref, names):
    for name in names:
        e = _rel(g[name], ref[name])
        assert e <= TAU, f"d{name}: max|err|/rms = {e:.3e}"


STRUCTURED = [
    # mode, dtype, dk, dv, H, T, S0
    ("gdn", "bf16", 128, 128, 2, 100, True),
    ("gdn", "f32", 64, 32, 2, 70, False),
    ("gdn", "f32", 32, 64, 1, 5, True),
    ("hdla", "bf16", 128, 128, 2, 50, True),
    ("hdla", "f32", 32, 32, 1, 33, False),
]


@pytest.mark.parametrize("mode,dtype,dk,dv,H,T,s0", STRUCTURED)
def test_backward_structured_matches_oracle(sdl, mode, dtype, dk, dv, H, T, s0):
    w = workloads.Workload(90, f"bwd_{mode}", mode, dtype, 1, 1, 0, dk, dv, 1 if mode == "gdn" else 2, 1, 64, s0)
    inp = workloads.generate(w, heads=[(0, h) for h in range(H)], T=T)
    rng = np.random.default_rng(5)
    do = rng.standard_normal((1, H, T, dv)).astype(np.float32)
    dST = rng.standard_normal((1, H, dk, dv)).astype(np.float32)
    g = _run(sdl, mode, dtype, inp, do, dST)
    ref = oracle.backward_inputs(inp, do, dST)
    _check(g, ref, ["q", "k", "v", "decay", "beta"] + (["S0"] if s0 else []))
    if not s0:
        _check(g, ref, ["S0"])


@pytest.mark.parametrize("dtype,dk,dv,r,p,T", [("f32", 64, 64, 4, 2, 40), ("f32", 32, 32, 1, 0, 21),
                                                ("bf16", 64, 128, 2, 1, 37), ("f32", 128, 64, 3, 2, 19),
                                                ("f32", 32, 32, 8, 8, 13)])
def test_backward_generic_matches_oracle(sdl, dtype, dk, dv, r, p, T):
    from test_parity_gpu import W, gen_generic
    w = W("generic", dtype, dk, dv, r, p)
    inp = gen_generic(w, 2, T, seed=300 + r)
    inp["S0"] = (0.2 * np.random.default_rng(4).standard_normal((1, 2, dk, dv))).astype(np.float32)
    if p == 0:
        inp["K"] = inp["V"] = None
    rng = np.random.default_rng(6)
    do = rng.standard_normal((1, 2, T, dv)).astype(np.float32)
    dST = rng.standard_normal((1, 2, dk, dv)).astype(np.float32)
    g = _run(sdl, "generic", dtype, inp, do, dST)
    Vd = inp["V"] if inp["V"] is not None else np.zeros((1, 2, T, 0, dv))
    Kd = inp["K"] if inp["K"] is not None else np.zeros((1, 2, T, 0, dk))
    ref = oracle.backward("generic", inp["q"], decay=inp["decay"], A=inp["A"], Bm=inp["Bm"], K=Kd, V=Vd,
                          S0=inp["S0"], do=do, dST=dST)
    _check(g, ref, ["q", "decay", "A", "Bm", "S0"] + (["K", "V"] if p else []))


def test_backward_without_final_state_gradient(sdl):
    """dST = None is the zero gradient."""
    w = workloads.Workload(91, "bwd_gdn", "gdn", "bf16", 1, 1, 0, 128, 128, 1, 1, 64, True)
    inp = workloads.generate(w, heads=[(0, 0)], T=64)
    do = np.random.default_rng(8).standard_normal((1, 1, 64, 128)).astype(np.float32)
    g = _run(sdl, "gdn", "bf16", inp, do, None)
    ref = oracle.backward_inputs(inp, do, None)
    _check(g, ref, ["q", "k", "v", "decay", "beta", "S0"])


def test_backward_full_size_workload_sampled_heads(sdl):
    """The backward workload the benchmark times, at full size (Gated DeltaNet bf16 B8 H16 T8192 d128), in one call
    over every head: every gradient finite, and two sampled heads compared with the float64 reverse mode over the
    whole sequence."""
    import torch
    w = workloads.WORKLOADS[2]
    inp = workloads.generate(w)
    rng = np.random.default_rng(21)
    do = rng.standard_normal((w.B, w.H, w.T, w.dv), dtype=np.float32)
    dST = rng.standard_normal((w.B, w.H, w.dk, w.dv), dtype=np.float32)
    d = lambda x, t: None if x is None else torch.from_numpy(np.ascontiguousarray(x)).to("cuda").to(t)
    bw = sdl.Backward("gdn", torch.bfloat16, w.B, w.H, w.T, w.dk, w.dv)
    g = bw(dO=d(do, torch.float32), dST=d(dST, torch.float32), q=d(inp["q"], torch.bfloat16),
           k=d(inp["k"], torch.bfloat16), v=d(inp["v"], torch.bfloat16), decay=d(inp["decay"], torch.float32),
           beta=d(inp["beta"], torch.float32), S0=d(inp["S0"], torch.float32))
    torch.cuda.synchronize()
    for name, x in g.items():
        if x is not None:
            assert bool(torch.isfinite(x).all()), f"d{name} not finite"
    pairs = [(0, 0), (7, 9)]
    sub = workloads.generate(w, heads=pairs)
    idx = (np.array([b for b, _ in pairs]), np.array([h for _, h in pairs]))
    ref = oracle.backward_inputs(sub, do[idx][None], dST[idx][None])
    for i, (b, h) in enumerate(pairs):
        for name in ("q", "k", "v", "decay", "beta", "S0"):
            e = _rel(g[name][b, h].double().cpu().numpy(), ref[name][0, i])
            assert e <= TAU, f"head {(b, h)} d{name}: max|err|/rms = {e:.3e}"
