"""HLA's query-gated composition (dplr_hla_forward) against the float64 oracle (oracle.hla).

Whole small problems, compared element by element: max |err| <= TAU * RMS of the oracle's output. The GPU path
composes the exact chunk maps in fp32 from exact inputs (bf16 values upcast), and the gated composition either in
fp32 (CUDA cores) or, for dk = dv = 128, on the tensor cores with bf16 hi + lo operands (~16 significant bits);
TAU = 1e-3 allows for the rounding of those products (the measured errors sit near 1e-6 to 1e-5).
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


def gates(H, T, L, seed, scale=2.0):
    """Synthetic gates in (0, 1): sigmoid of N(-1, scale) per (query, chunk)."""
    N = (T + L - 1) // L
    z = np.random.default_rng(seed).standard_normal((1, H, T, N)) * scale - 1.0
    return (1.0 / (1.0 + np.exp(-z))).astype(np.float32)


CASES = [
    # dtype, dk, dv, H, T, L, theta  (dk = dv = 128: the tensor-core composition and gated passes)
    ("bf16", 128, 128, 2, 700, 256, 0.1),
    ("f32", 128, 128, 1, 450, 128, 0.1),
    ("bf16", 128, 128, 1, 266, 256, 0.0),    # the last chunk a single ragged block
    ("bf16", 128, 128, 2, 50, 256, 0.1),     # one chunk of one block: no history
    ("bf16", 128, 128, 2, 300, 64, 0.0),
    ("f32", 128, 128, 1, 830, 64, 0.5),
    ("f32", 64, 64, 2, 500, 128, 0.1),
    ("f32", 64, 128, 1, 257, 256, 0.5),
    ("bf16", 128, 64, 1, 64, 64, 0.1),
]


@pytest.mark.parametrize("dtype,dk,dv,H,T,L,theta", CASES)
def test_hla_matches_oracle(sdl, dtype, dk, dv, H, T, L, theta):
    import torch
    w = workloads.Workload(89, "hla_gdn", "gdn", dtype, 1, 1, 0, dk, dv, 1, 1, 64, False)
    inp = workloads.generate(w, heads=[(0, h) for h in range(H)], T=T)
    W = gates(H, T, L, seed=T + L)
    dt = torch.bfloat16 if dtype == "bf16" else torch.float32
    d = lambda x, t: torch.from_numpy(np.ascontiguousarray(x)).to("cuda").to(t)
    f = sdl.HLA(dt, 1, H, T, dk, dv, L)
    o = f(d(inp["q"], dt), d(inp["k"], dt), d(inp["v"], dt), d(inp["decay"], torch.float32),
          d(inp["beta"], torch.float32), d(W, torch.float32), theta)
    torch.cuda.synchronize()
    ref = oracle.hla(inp["q"], inp["k"], inp["v"], inp["decay"], inp["beta"], W, L, theta)
    e = _rel(o.double().cpu().numpy(), ref)
    assert e <= TAU, f"max|err|/rms = {e:.3e}"


def test_hla_all_gates_one_is_the_forward(sdl):
    """With every gate 1 the composition is the plain GDN recurrence: dplr_hla_forward equals dplr_la_forward."""
    import torch
    w = workloads.Workload(88, "hla_gdn", "gdn", "bf16", 1, 1, 0, 128, 128, 1, 1, 64, False)
    H, T, L = 2, 512, 128
    inp = workloads.generate(w, heads=[(0, h) for h in range(H)], T=T)
    d = lambda x, t: torch.from_numpy(np.ascontiguousarray(x)).to("cuda").to(t)
    args = [d(inp["q"], torch.bfloat16), d(inp["k"], torch.bfloat16), d(inp["v"], torch.bfloat16),
            d(inp["decay"], torch.float32), d(inp["beta"], torch.float32)]
    o = sdl.HLA(torch.bfloat16, 1, H, T, 128, 128, L)(*args, d(np.ones((1, H, T, T // L)), torch.float32), 0.1)
    f = sdl.Forward("gdn", torch.bfloat16, 1, H, T, 128, 128)
    o2, _ = f(q=args[0], k=args[1], v=args[2], decay=args[3], beta=args[4])
    torch.cuda.synchronize()
    ref, _ = oracle.forward_inputs(inp)
    assert _rel(o.double().cpu().numpy(), ref) <= TAU
    assert _rel(o.double().cpu().numpy(), o2.double().cpu().numpy()) <= 2e-2


def test_hla_paths(sdl):
    """dk = dv = 128 takes the tensor-core gated pass (up to 256 chunks); other sizes the fp32 pass."""
    import torch
    p = lambda dk, dv, T, L: sdl.dplr_hla_path(sdl.make_desc("gdn", torch.bfloat16, 1, 2, T, dk, dv), L)
    assert p(128, 128, 4096, 256) == "hla_gated_tcgen05"
    assert p(128, 128, 16384, 64) == "hla_gated_tcgen05"
    assert p(128, 128, 16448, 64) == "hla_gated_fp32"      # 257 chunks
    assert p(64, 64, 4096, 256) == "hla_gated_fp32"
    assert p(128, 64, 4096, 256) == "hla_gated_fp32"
    assert p(128, 128, 4096, 100) == ""


def test_hla_tensor_core_pass_timeout_returns_and_reports(sdl):
    """The tensor-core gated pass's waits, limited to 1000 cycles, end the launch with DPLR_ERR_TIMEOUT in the
    status word; with the default limit the same context gives a correct composition."""
    import torch
    w = workloads.Workload(87, "hla_gdn", "gdn", "bf16", 1, 1, 0, 128, 128, 1, 1, 64, False)
    H, T, L = 2, 1024, 128
    inp = workloads.generate(w, heads=[(0, h) for h in range(H)], T=T)
    W = gates(H, T, L, seed=5)
    d = lambda x, t: torch.from_numpy(np.ascontiguousarray(x)).to("cuda").to(t)
    args = [d(inp["q"], torch.bfloat16), d(inp["k"], torch.bfloat16), d(inp["v"], torch.bfloat16),
            d(inp["decay"], torch.float32), d(inp["beta"], torch.float32), d(W, torch.float32), 0.1]
    f = sdl.HLA(torch.bfloat16, 1, H, T, 128, 128, L)
    assert f.path == "hla_gated_tcgen05"
    sdl.dplr_la_set_wait_limit(1000)
    try:
        f(*args)
        torch.cuda.synchronize()
        assert f.device_status() == sdl.dplr.DPLR_ERR_TIMEOUT
    finally:
        sdl.dplr_la_set_wait_limit(0)
    o = f(*args)
    torch.cuda.synchronize()
    assert f.device_status() == sdl.DPLR_OK
    ref = oracle.hla(inp["q"], inp["k"], inp["v"], inp["decay"], inp["beta"], W, L, 0.1)
    assert _rel(o.double().cpu().numpy(), ref) <= TAU


def test_hla_full_size_gates_one_and_zero(sdl):
    """The HLA workload the benchmark times, at full size (Gated DeltaNet bf16 B1 H16 T4096 d128, L = 256), through
    two properties that hold at any size. With every gate 1 the composition is the plain recurrence: two sampled
    heads against the float64 forward, every head against the fused forward. With every gate 0 no history enters,
    so each 256-token chunk starts from a zero state: every head against the fused forward of the chunks taken as
    separate sequences."""
    import torch
    H, T, L = 16, 4096, 256
    N = T // L
    w = workloads.Workload(98, "hla_gdn_bf16_b1h16", "gdn", "bf16", 1, H, T, 128, 128, 1, 1, 64, False)
    inp = workloads.generate(w)
    d = lambda x, t: torch.from_numpy(np.ascontiguousarray(x)).to("cuda").to(t)
    args = [d(inp["q"], torch.bfloat16), d(inp["k"], torch.bfloat16), d(inp["v"], torch.bfloat16),
            d(inp["decay"], torch.float32), d(inp["beta"], torch.float32)]
    f = sdl.HLA(torch.bfloat16, 1, H, T, 128, 128, L)
    assert f.path == "hla_gated_tcgen05"
    o1 = f(*args, torch.ones(1, H, T, N, device="cuda"), 0.1).clone()
    o0 = f(*args, torch.zeros(1, H, T, N, device="cuda"), 0.1).clone()
    fwd = sdl.Forward("gdn", torch.bfloat16, 1, H, T, 128, 128)
    of, _ = fwd(q=args[0], k=args[1], v=args[2], decay=args[3], beta=args[4])
    of = of.clone()
    chunks = lambda x: x.reshape(1, H * N, L, *x.shape[3:]).contiguous()
    fl = sdl.Forward("gdn", torch.bfloat16, 1, H * N, L, 128, 128)
    ol, _ = fl(q=chunks(args[0]), k=chunks(args[1]), v=chunks(args[2]), decay=chunks(args[3]), beta=chunks(args[4]))
    torch.cuda.synchronize()
    assert bool(torch.isfinite(o1).all()) and bool(torch.isfinite(o0).all())
    host = lambda x: x.double().cpu().numpy()
    assert _rel(host(o1), host(of)) <= 2e-2
    assert _rel(host(o0), host(ol.reshape(1, H, T, 128))) <= 2e-2
    pairs = [(0, 0), (0, 11)]
    ref, _ = oracle.forward_inputs(workloads.generate(w, heads=pairs))
    for i, (b, h) in enumerate(pairs):
        e = _rel(host(o1[b, h]), ref[0, i])
        assert e <= TAU, f"head {(b, h)}: max|err|/rms = {e:.3e}"
