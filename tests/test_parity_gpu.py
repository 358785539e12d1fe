"""Parity of the CUDA path (through the C ABI) with the float64 oracle.

Tolerance (stated with the workloads): max |o_gpu - o_ref| <= tau * RMS(o_ref), tau = 1e-4
for float32 inputs and 2e-2 for bf16 inputs with float32 state; the same bound is applied
to the final state S_T against RMS(S_T_ref). Both sides consume the same seeded inputs
(bf16 values upcast exactly for the oracle).
"""

import numpy as np
import pytest

import oracle
import workloads

pytestmark = pytest.mark.gpu

TAU = {"f32": 1e-4, "bf16": 2e-2}


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


def _to_dev(x, dtype):
    import torch
    if x is None:
        return None
    return torch.from_numpy(np.ascontiguousarray(x)).to("cuda").to(dtype)


def run_gpu(sdl, inp, S0=None, fwd=None):
    import torch
    w = inp["workload"]
    dt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    S0 = inp["S0"] if S0 is None else S0
    args = dict(q=_to_dev(inp["q"], dt), k=_to_dev(inp["k"], dt), v=_to_dev(inp["v"], dt),
                decay=_to_dev(inp["decay"], torch.float32), beta=_to_dev(inp["beta"], torch.float32),
                A=_to_dev(inp["A"], dt), Bm=_to_dev(inp["Bm"], dt), K=_to_dev(inp["K"], dt),
                V=_to_dev(inp["V"], dt), S0=_to_dev(S0, torch.float32))
    if fwd is None:
        fwd = sdl.Forward(w.mode, dt, inp["B"], inp["H"], inp["T"], w.dk, w.dv, w.r_ab, w.r_kv, w.chunk)
    o, ST = fwd(**args)
    torch.cuda.synchronize()
    return o.double().cpu().numpy(), ST.double().cpu().numpy()


def rel_err(a, ref):
    rms = float(np.sqrt(np.mean(ref ** 2))) if ref.size else 0.0
    if ref.size == 0:
        return 0.0
    return float(np.abs(a - ref).max()) / max(rms, 1e-30)


def check(inp, o, ST, S0=None, heads=None):
    w = inp["workload"]
    ref_inp = inp
    if S0 is not None:
        ref_inp = dict(inp)
        ref_inp["S0"] = S0
    o_ref, S_ref = oracle.forward_inputs(ref_inp)
    tau = TAU[w.dtype]
    eo, es = rel_err(o, o_ref), rel_err(ST, S_ref)
    assert np.isfinite(o).all() and np.isfinite(ST).all()
    assert eo <= tau, f"o: max|err|/rms = {eo:.3e} > {tau}"
    assert es <= tau, f"S_T: max|err|/rms = {es:.3e} > {tau}"
    return eo, es


def W(mode, dtype, dk, dv, r=None, p=None, s0=False):
    r = r if r is not None else {"gdn": 1, "hdla": 2}.get(mode, 1)
    p = p if p is not None else 1
    return workloads.Workload(99, f"{mode}_{dtype}_{dk}x{dv}_r{r}p{p}", mode, dtype, 1, 1, 0, dk, dv, r, p, 64, s0)


def gen_generic(w, H, T, seed):
    """Generic-mode inputs of arbitrary rank in the generator's recipe (Q-factor U_t)."""
    rng = np.random.default_rng(seed)
    f32 = np.float32
    q = rng.standard_normal((1, H, T, w.dk), dtype=f32)
    decay = (-np.logaddexp(0, -(rng.standard_normal((1, H, T, w.dk)) + 2))).astype(f32)
    r, p = w.r_ab, w.r_kv
    beta = 2 / (1 + np.exp(-rng.standard_normal((1, H, T, r))))
    g = rng.standard_normal((1, H, T, w.dk, r))
    U = np.linalg.qr(g.reshape(-1, w.dk, r), mode="reduced")[0].reshape(g.shape)
    A = (np.exp(decay)[..., None] * U * beta[..., None, :]).transpose(0, 1, 2, 4, 3).astype(f32)
    Bm = U.transpose(0, 1, 2, 4, 3).astype(f32)
    K = (rng.standard_normal((1, H, T, p, w.dk)) / 8).astype(f32) if p else None
    V = (rng.standard_normal((1, H, T, p, w.dv)) / 8).astype(f32) if p else None
    out = dict(q=q, decay=decay, A=A, Bm=Bm, K=K, V=V, k=None, v=None, beta=None, S0=None)
    if w.dtype == "bf16":
        for key in ("q", "A", "Bm", "K", "V"):
            if out[key] is not None:
                out[key] = workloads.round_to_bf16(out[key])
    out.update(workload=w, B=1, H=H, T=T)
    return out


SMALL_STRUCTURED = [
    # mode, dtype, dk, dv, H, T, s0
    ("gdn", "f32", 32, 32, 2, 256, False),
    ("gdn", "f32", 128, 64, 2, 1, True),
    ("gdn", "f32", 64, 128, 3, 200, True),
    ("gdn", "f32", 128, 128, 1, 300, True),   # two-stage path with its largest scan staging (64-token blocks, d = 128)
    ("gdn", "bf16", 128, 128, 3, 200, False),
    ("gdn", "bf16", 32, 64, 2, 5, True),
    ("hdla", "bf16", 128, 128, 2, 130, True),
    ("hdla", "f32", 64, 32, 2, 97, True),
    ("hdla", "f32", 128, 128, 1, 333, False),
    ("hdla", "bf16", 32, 128, 4, 64, True),
]


@pytest.mark.parametrize("mode,dtype,dk,dv,H,T,s0", SMALL_STRUCTURED)
def test_structured_small(sdl, mode, dtype, dk, dv, H, T, s0):
    w = W(mode, dtype, dk, dv, s0=s0)
    inp = workloads.generate(w, heads=[(0, h) for h in range(H)], T=T)
    o, ST = run_gpu(sdl, inp)
    check(inp, o, ST)


SMALL_GENERIC = [
    # dtype, dk, dv, r, p, H, T
    ("f32", 64, 64, 4, 2, 2, 100),
    ("f32", 32, 32, 1, 0, 1, 50),
    ("f32", 32, 32, 8, 8, 1, 40),
    ("bf16", 32, 128, 3, 1, 2, 77),
    ("f32", 128, 64, 2, 3, 1, 129),
    ("bf16", 128, 128, 4, 2, 1, 64),
]


@pytest.mark.parametrize("dtype,dk,dv,r,p,H,T", SMALL_GENERIC)
def test_generic_small(sdl, dtype, dk, dv, r, p, H, T):
    w = W("generic", dtype, dk, dv, r, p)
    inp = gen_generic(w, H, T, seed=1000 + r * 10 + p)
    S0 = (0.2 * np.random.default_rng(5).standard_normal((1, H, dk, dv))).astype(np.float32)
    inp["S0"] = S0
    o, ST = run_gpu(sdl, inp)
    check(inp, o, ST)


GENERIC_TC = [
    # dtype, r, p, H, T  (dk = dv = 64: the tensor-core chunk kernel, 32-token WY blocks)
    ("f32", 4, 2, 2, 100),    # several blocks and a ragged last one
    ("f32", 1, 0, 1, 50),     # no write term
    ("f32", 3, 1, 2, 77),     # 96 factor rows: zero-padded tiles
    ("f32", 2, 2, 1, 32),     # exactly one block
    ("f32", 4, 2, 1, 1),      # one token
    ("f32", 4, 1, 3, 33),     # one token past a block
    ("f32", 1, 2, 1, 129),
    ("bf16", 4, 2, 2, 200),
    ("f32", 1, 0, 2, 8192),   # the generic workload's sequence length at other ranks
    ("f32", 3, 1, 2, 8192),
]


@pytest.mark.parametrize("dtype,r,p,H,T", GENERIC_TC)
def test_generic_tensor_core_path(sdl, dtype, r, p, H, T):
    w = W("generic", dtype, 64, 64, r, p)
    assert sdl.dplr_la_path(sdl.make_desc("generic", dtype, 1, H, T, 64, 64, r, p)) == "generic_tcgen05"
    inp = gen_generic(w, H, T, seed=2000 + 10 * r + p)
    inp["S0"] = (0.2 * np.random.default_rng(6).standard_normal((1, H, 64, 64))).astype(np.float32)
    o, ST = run_gpu(sdl, inp)
    check(inp, o, ST)


def test_generic_tensor_core_slow_decay(sdl):
    """Decay close to one (log-decay -0.005 per channel and token): the block's factors span e^{+-0.08} only, and
    the chunk maps are far from contracting, so rounding in P_j carries over many blocks."""
    w = W("generic", "f32", 64, 64, 4, 2)
    inp = gen_generic(w, 1, 600, seed=2100)
    inp["decay"] = np.full_like(inp["decay"], -0.005)
    lam = np.exp(inp["decay"].astype(np.float64))[..., None, :]
    inp["A"] = (lam * inp["Bm"].astype(np.float64) * 0.5).astype(np.float32)   # D - A B^T = Diag(lambda)(I - U U^T / 2)
    o, ST = run_gpu(sdl, inp)
    check(inp, o, ST)


def test_config0_full(sdl):
    inp = workloads.generate(0)
    o, ST = run_gpu(sdl, inp)
    check(inp, o, ST)


def test_empty_sequence_returns_initial_state(sdl):
    w = W("hdla", "bf16", 64, 64, s0=True)
    inp = workloads.generate(w, heads=[(0, 0), (0, 1)], T=0)
    o, ST = run_gpu(sdl, inp)
    assert o.shape == (1, 2, 0, 64)
    assert np.array_equal(ST, inp["S0"].astype(np.float64))


def test_state_carry_across_calls(sdl):
    """forward(T1) then forward(T2, S0 = S_T1) equals forward(T1 + T2) (affine closure)."""
    w = W("hdla", "bf16", 128, 128, s0=True)
    inp = workloads.generate(w, heads=[(0, 0), (0, 1)], T=300)
    o_full, S_full = run_gpu(sdl, inp)

    def part(t0, t1):
        d = dict(inp)
        for key in ("q", "k", "v", "decay", "beta"):
            d[key] = np.ascontiguousarray(inp[key][:, :, t0:t1])
        d["T"] = t1 - t0
        return d
    a = part(0, 150)
    oa, Sa = run_gpu(sdl, a)
    b = part(150, 300)
    ob, Sb = run_gpu(sdl, b, S0=Sa.astype(np.float32))
    o_ref, S_ref = oracle.forward_inputs(inp)
    assert rel_err(np.concatenate([oa, ob], axis=2), o_ref) <= TAU["bf16"]
    assert rel_err(Sb, S_ref) <= TAU["bf16"]
    assert rel_err(np.concatenate([oa, ob], axis=2), o_full) <= TAU["bf16"]


def test_stage_calls_match_forward_and_are_deterministic(sdl):
    """The two-stage entry points and the forward (fused kernel here) agree within tolerance;
    each is bitwise deterministic from call to call."""
    import torch
    w = W("gdn", "bf16", 128, 128, s0=True)
    inp = workloads.generate(w, heads=[(0, 0), (0, 1), (0, 2)], T=257)
    dt = torch.bfloat16
    fwd = sdl.Forward("gdn", dt, 1, 3, 257, 128, 128)
    args = dict(q=_to_dev(inp["q"], dt), k=_to_dev(inp["k"], dt), v=_to_dev(inp["v"], dt),
                decay=_to_dev(inp["decay"], torch.float32), beta=_to_dev(inp["beta"], torch.float32))
    S0 = _to_dev(inp["S0"], torch.float32)
    o1, S1 = [x.clone() for x in fwd(**args, S0=S0)]
    o2, S2 = [x.clone() for x in fwd(**args, S0=S0)]
    fwd.chunk_maps(**args)
    o3, S3 = [x.clone() for x in fwd.state_scan(S0)]
    fwd.chunk_maps(**args)
    o4, S4 = [x.clone() for x in fwd.state_scan(S0)]
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(S1, S2)
    assert torch.equal(o3, o4) and torch.equal(S3, S4)
    a = lambda x: x.double().cpu().numpy()
    assert rel_err(a(o1), a(o3)) <= TAU["bf16"] and rel_err(a(S1), a(S3)) <= TAU["bf16"]
    assert fwd.device_status() == 0


@pytest.mark.parametrize("B,H,T", [(1, 2, 1), (1, 2, 63), (1, 2, 64), (1, 2, 65), (2, 3, 191), (1, 1, 1024)])
def test_fused_kernel_edges(sdl, B, H, T):
    """The fused GDN kernel on sequences shorter than a chunk, exactly one chunk, one past it,
    several heads with a ragged tail, and a longer run (S0 nonzero throughout)."""
    w = W("gdn", "bf16", 128, 128, s0=True)
    assert sdl.dplr_la_kernel_count(sdl.make_desc("gdn", "bf16", B, H, T, 128, 128)) == 1
    inp = workloads.generate(w, heads=[(b, h) for b in range(B) for h in range(H)], T=T)
    o, ST = run_gpu(sdl, inp)
    check(inp, o, ST)


def test_fused_kernel_empty_sequence(sdl):
    w = W("gdn", "bf16", 128, 128, s0=True)
    inp = workloads.generate(w, heads=[(0, 0), (0, 1)], T=0)
    o, ST = run_gpu(sdl, inp)
    assert o.shape == (1, 2, 0, 128)
    assert np.array_equal(ST, inp["S0"].astype(np.float64))


@pytest.mark.parametrize("B,H,T", [(1, 2, 1), (1, 2, 63), (1, 2, 64), (1, 2, 65), (2, 3, 191), (1, 1, 1024)])
def test_hdla_tensor_core_path_edges(sdl, B, H, T):
    """The tensor-core HDLA stages (bf16, d = 128) on sequences shorter than a chunk, exactly one
    chunk, one past it, several heads with a ragged tail, and a longer run (S0 nonzero throughout)."""
    w = W("hdla", "bf16", 128, 128, s0=True)
    d = sdl.make_desc("hdla", "bf16", B, H, T, 128, 128)
    assert sdl.dplr_la_kernel_count(d) == 2
    inp = workloads.generate(w, heads=[(b, h) for b in range(B) for h in range(H)], T=T)
    o, ST = run_gpu(sdl, inp)
    check(inp, o, ST)


def test_hdla_tensor_core_path_empty_sequence(sdl):
    w = W("hdla", "bf16", 128, 128, s0=True)
    inp = workloads.generate(w, heads=[(0, 0), (0, 1)], T=0)
    o, ST = run_gpu(sdl, inp)
    assert o.shape == (1, 2, 0, 128)
    assert np.array_equal(ST, inp["S0"].astype(np.float64))


def test_hdla_stage_calls_match_forward_and_are_deterministic(sdl):
    """On the tensor-core HDLA path, dplr_la_chunk_maps then dplr_la_state_scan give the same bits as
    dplr_la_forward, call after call, and the status word stays clear."""
    import torch
    w = W("hdla", "bf16", 128, 128, s0=True)
    inp = workloads.generate(w, heads=[(0, 0), (0, 1), (0, 2)], T=257)
    dt = torch.bfloat16
    fwd = sdl.Forward("hdla", dt, 1, 3, 257, 128, 128)
    assert fwd.ws_bytes == fwd.stage_ws_bytes
    args = dict(q=_to_dev(inp["q"], dt), k=_to_dev(inp["k"], dt), v=_to_dev(inp["v"], dt),
                decay=_to_dev(inp["decay"], torch.float32), beta=_to_dev(inp["beta"], torch.float32))
    S0 = _to_dev(inp["S0"], torch.float32)
    o1, S1 = [x.clone() for x in fwd(**args, S0=S0)]
    o2, S2 = [x.clone() for x in fwd(**args, S0=S0)]
    fwd.chunk_maps(**args)
    o3, S3 = [x.clone() for x in fwd.state_scan(S0)]
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(S1, S2)
    assert torch.equal(o1, o3) and torch.equal(S1, S3)
    assert fwd.device_status() == 0
    check(inp, o1.double().cpu().numpy(), S1.double().cpu().numpy())


def test_fused_path_selection(sdl):
    """GDN with bf16 inputs at d=128 runs one fused kernel with a status-word workspace; others two stages."""
    d = sdl.make_desc("gdn", "bf16", 8, 16, 8192, 128, 128)
    assert sdl.dplr_la_kernel_count(d) == 1 and sdl.dplr_la_workspace_size(d) == 256
    d = sdl.make_desc("gdn", "f32", 1, 2, 256, 32, 32)
    assert sdl.dplr_la_kernel_count(d) == 2
    assert sdl.dplr_la_workspace_size(d) == sdl.dplr_la_stage_workspace_size(d) > 0
    # HDLA bf16 d = 128: the tensor-core stages, whose workspace holds per chunk P_j (bf16 128 x 128),
    # c_j (fp32 128 x 128) and Q'_j (bf16 hi and lo, 64 x 128 each) after the status word
    d = sdl.make_desc("hdla", "bf16", 4, 16, 4096, 128, 128)
    assert sdl.dplr_la_kernel_count(d) == 2
    assert sdl.dplr_la_workspace_size(d) == 256 + 64 * 64 * (32768 + 65536 + 32768)


# ---------------------------------------------------------------------------
# Full-size workloads, in the launch configuration the benchmark times: every head
# is computed on the GPU; sampled heads are compared with the oracle over the whole
# sequence, and every output is checked finite.
# ---------------------------------------------------------------------------

SAMPLED = {1: [(0, 0), (3, 15)], 2: [(0, 0), (7, 9)], 3: [(0, 0), (1, 7)], 4: [(0, 0), (0, 11)]}


@pytest.mark.parametrize("wid", [1, 2, 3, 4])
def test_full_size_workload_sampled_heads(sdl, wid):
    w = workloads.WORKLOADS[wid]
    inp = workloads.generate(w)
    o, ST = run_gpu(sdl, inp)
    assert np.isfinite(o).all() and np.isfinite(ST).all()
    pairs = SAMPLED[wid]
    sub = workloads.generate(w, heads=pairs)
    o_ref, S_ref = oracle.forward_inputs(sub)
    tau = TAU[w.dtype]
    for i, (b, h) in enumerate(pairs):
        eo = rel_err(o[b, h], o_ref[0, i])
        es = rel_err(ST[b, h], S_ref[0, i])
        assert eo <= tau, f"workload {wid} head {(b, h)}: o err {eo:.3e}"
        assert es <= tau, f"workload {wid} head {(b, h)}: S_T err {es:.3e}"


@pytest.mark.parametrize("mode,groups,slots,s0", [("gdn", 4, 2, True), ("gdn", 8, 8, False), ("hdla", 2, 1, True)])
def test_forward_host_matches_device_forward(sdl, mode, groups, slots, s0):
    """dplr_la_forward_host (host buffers, heads split into groups through a ring of staging
    slots) gives the same bits as dplr_la_forward on device buffers, on two calls in a row."""
    import torch
    w = W(mode, "bf16", 128, 128, s0=s0)
    B, H, T = 2, 4, 200
    inp = workloads.generate(w, heads=[(b, h) for b in range(B) for h in range(H)], T=T)
    host = {}
    for key in ("q", "k", "v", "decay", "beta", "S0"):
        x = inp[key]
        if x is None:
            host[key] = None
            continue
        x = np.ascontiguousarray(x).reshape((B, H) + x.shape[2:])
        t = torch.from_numpy(x)
        host[key] = (t.to(torch.bfloat16) if key in ("q", "k", "v") else t).pin_memory()
    dev = {k_: (None if t is None else t.to("cuda")) for k_, t in host.items()}
    ref = sdl.Forward(mode, torch.bfloat16, B, H, T, 128, 128)
    o_ref, S_ref = [x.clone() for x in ref(**dev)]
    fh = sdl.ForwardHost(mode, torch.bfloat16, B, H, T, 128, 128, groups=groups, slots=slots)
    for _ in range(2):
        fh.o.fill_(float("nan"))
        fh.S_T.fill_(float("nan"))
        o, S = fh(**host)
        torch.cuda.current_stream().synchronize()
        assert torch.equal(o, o_ref.cpu()) and torch.equal(S, S_ref.cpu())


@pytest.mark.parametrize("mode,T,segments,slots,s0", [("gdn", 200, 3, 2, True), ("gdn", 1000, 4, 2, False),
                                                       ("gdn", 64, 8, 8, True), ("hdla", 300, 2, 1, True),
                                                       ("gdn", 0, 4, 2, True)])
def test_forward_host_seq_matches_device_forward(sdl, mode, T, segments, slots, s0):
    """dplr_la_forward_host_seq (host buffers, the sequence split into segments whose forwards carry
    the state on the device) gives dplr_la_forward's result: the same bits on the fused GDN kernel,
    within 1e-5 of the RMS on the HDLA stages; on two calls in a row."""
    import torch
    w = W(mode, "bf16", 128, 128, s0=s0)
    B, H = 2, 3
    inp = workloads.generate(w, heads=[(b, h) for b in range(B) for h in range(H)], T=max(T, 1))
    host = {}
    for key in ("q", "k", "v", "decay", "beta", "S0"):
        x = inp[key]
        if x is None:
            host[key] = None
            continue
        x = np.ascontiguousarray(x).reshape((B, H) + x.shape[2:])
        if key != "S0":
            x = np.ascontiguousarray(x[:, :, :T])
        t = torch.from_numpy(x)
        host[key] = (t.to(torch.bfloat16) if key in ("q", "k", "v") else t).pin_memory()
    dev = {k_: (None if t is None else t.to("cuda")) for k_, t in host.items()}
    ref = sdl.Forward(mode, torch.bfloat16, B, H, T, 128, 128)
    o_ref, S_ref = [x.clone().cpu() for x in ref(**dev)]
    fh = sdl.ForwardHostSeq(mode, torch.bfloat16, B, H, T, 128, 128, segments=segments, slots=slots)
    for _ in range(2):
        fh.o.fill_(float("nan"))
        fh.S_T.fill_(float("nan"))
        o, S = fh(**host)
        torch.cuda.current_stream().synchronize()
        if mode == "gdn":
            assert torch.equal(o, o_ref) and torch.equal(S, S_ref)
        else:
            for x, y in ((o, o_ref), (S, S_ref)):
                scale = float(y.double().pow(2).mean().sqrt()) or 1.0
                assert float((x.double() - y.double()).abs().max()) <= 1e-5 * scale


@pytest.mark.parametrize("dtype,r,p,T,segments", [("f32", 4, 2, 700, 3), ("bf16", 2, 1, 260, 2), ("f32", 3, 0, 130, 2)])
def test_forward_host_seq_generic_matches_device_forward(sdl, dtype, r, p, T, segments):
    """dplr_la_forward_host_seq in the generic mode (the tensor-core generic stages at d = 64, and a rank-3
    case without K and V on the fp32 stages) gives dplr_la_forward's result within 1e-5 of the RMS."""
    import torch
    w = workloads.Workload(96, "generic_host_seq", "generic", dtype, 1, 2, T, 64, 64, r, p, 64, False)
    inp = gen_generic(w, 2, T, seed=T + r)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    host = {}
    for key in ("q", "decay", "A", "Bm", "K", "V"):
        x = inp[key]
        if x is None:
            host[key] = None
            continue
        t = torch.from_numpy(np.ascontiguousarray(x))
        host[key] = (t.to(tdt) if key != "decay" else t).pin_memory()
    dev = {k_: (None if t is None else t.to("cuda")) for k_, t in host.items()}
    ref = sdl.Forward("generic", tdt, 1, 2, T, 64, 64, r, p)
    o_ref, S_ref = [x.clone().cpu() for x in ref(**dev)]
    fh = sdl.ForwardHostSeq("generic", tdt, 1, 2, T, 64, 64, r, p, segments=segments, slots=2)
    o, S = fh(**host)
    torch.cuda.current_stream().synchronize()
    for x, y in ((o, o_ref), (S, S_ref)):
        scale = float(y.double().pow(2).mean().sqrt()) or 1.0
        assert float((x.double() - y.double()).abs().max()) <= 1e-5 * scale
