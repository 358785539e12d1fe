"""The one-token decode step (dplr_la_decode_step) against the float64 oracle.

A sequence decoded token by token, carrying the state, must reproduce the serial recurrence:
every output o_t and the final state. The step computes in fp32 from exact inputs (bf16 values
upcast), so the fp32 tolerance applies to every input type: max |err| <= 1e-4 * RMS. A decode
continued from the state of a chunked forward (dplr_la_forward) must match the oracle over the
whole sequence within the chunked path's tolerance.
"""

import numpy as np
import pytest

import oracle
import workloads

pytestmark = pytest.mark.gpu

TAU_STEP = 1e-4
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


def _rel(a, ref):
    return float(np.abs(a - ref).max() / max(np.sqrt(np.mean(ref ** 2)), 1e-30))


def _token(inp, key, t):
    x = inp[key]
    return None if x is None else np.ascontiguousarray(x[:, :, t:t + 1])


def _decode(sdl, inp, mode, dtype, S0, t0=0):
    import torch
    w = inp["workload"]
    dt = torch.bfloat16 if dtype == "bf16" else torch.float32
    B, H, T = inp["B"], inp["H"], inp["T"]
    dev = lambda x, d: None if x is None else torch.from_numpy(x).to("cuda").to(d)
    r_ab = inp["A"].shape[3] if inp["A"] is not None else None
    r_kv = inp["K"].shape[3] if inp["K"] is not None else (0 if mode == "generic" else None)
    step = sdl.Decode(mode, dt, B, H, w.dk, w.dv, r_ab, r_kv,
                      S0=None if S0 is None else torch.from_numpy(np.ascontiguousarray(S0)).to("cuda"))
    outs = []
    for t in range(t0, T):
        o = step(q=dev(_token(inp, "q", t), dt), k=dev(_token(inp, "k", t), dt), v=dev(_token(inp, "v", t), dt),
                 decay=dev(_token(inp, "decay", t), torch.float32), beta=dev(_token(inp, "beta", t), torch.float32),
                 A=dev(_token(inp, "A", t), dt), Bm=dev(_token(inp, "Bm", t), dt), K=dev(_token(inp, "K", t), dt),
                 V=dev(_token(inp, "V", t), dt))
        outs.append(o.double().cpu().numpy())
    torch.cuda.synchronize()
    return np.concatenate(outs, axis=2), step.S.double().cpu().numpy()


CASES = [
    # mode, dtype, dk, dv, H, T
    ("gdn", "bf16", 128, 128, 3, 9),
    ("gdn", "f32", 64, 32, 2, 7),
    ("hdla", "bf16", 128, 128, 2, 9),
    ("hdla", "f32", 32, 64, 2, 6),
]


@pytest.mark.parametrize("mode,dtype,dk,dv,H,T", CASES)
def test_decode_matches_the_recurrence(sdl, mode, dtype, dk, dv, H, T):
    w = workloads.Workload(93, f"dec_{mode}", mode, dtype, 1, 1, 0, dk, dv, 1 if mode == "gdn" else 2, 1, 64, True)
    inp = workloads.generate(w, heads=[(0, h) for h in range(H)], T=T)
    o, S = _decode(sdl, inp, mode, dtype, inp["S0"])
    o_ref, S_ref = oracle.forward_inputs(inp)
    assert _rel(o, o_ref) <= TAU_STEP and _rel(S, S_ref) <= TAU_STEP


@pytest.mark.parametrize("dtype,dk,dv,r,p", [("f32", 64, 64, 4, 2), ("bf16", 128, 32, 8, 8), ("f32", 32, 128, 1, 0)])
def test_decode_generic_matches_the_recurrence(sdl, dtype, dk, dv, r, p):
    from test_parity_gpu import W, gen_generic
    w = W("generic", dtype, dk, dv, r, p)
    inp = gen_generic(w, 2, 6, seed=77 + r)
    inp["S0"] = (0.2 * np.random.default_rng(3).standard_normal((1, 2, dk, dv))).astype(np.float32)
    o, S = _decode(sdl, inp, "generic", dtype, inp["S0"])
    o_ref, S_ref = oracle.forward_inputs(inp)
    assert _rel(o, o_ref) <= TAU_STEP and _rel(S, S_ref) <= TAU_STEP


@pytest.mark.parametrize("mode", ["gdn", "hdla"])
def test_decode_continues_a_chunked_forward(sdl, mode):
    """Prefill 130 tokens with dplr_la_forward (the tensor-core paths), then decode 6 more from its
    final state: the decoded outputs and the final state match the oracle over all 136 tokens."""
    import torch
    w = workloads.Workload(92, f"prefill_{mode}", mode, "bf16", 1, 1, 0, 128, 128, 1 if mode == "gdn" else 2, 1, 64,
                           True)
    T1, T2 = 130, 6
    inp = workloads.generate(w, heads=[(0, 0), (0, 1)], T=T1 + T2)
    pre = dict(inp)
    for key in ("q", "k", "v", "decay", "beta"):
        pre[key] = np.ascontiguousarray(inp[key][:, :, :T1])
    pre["T"] = T1
    dt = torch.bfloat16
    d = lambda x, t: torch.from_numpy(np.ascontiguousarray(x)).to("cuda").to(t)
    f = sdl.Forward(mode, dt, 1, 2, T1, 128, 128)
    _, S1 = f(q=d(pre["q"], dt), k=d(pre["k"], dt), v=d(pre["v"], dt), decay=d(pre["decay"], torch.float32),
              beta=d(pre["beta"], torch.float32), S0=d(inp["S0"], torch.float32))
    torch.cuda.synchronize()
    o2, S2 = _decode(sdl, inp, mode, "bf16", S1.cpu().numpy(), t0=T1)
    o_ref, S_ref = oracle.forward_inputs(inp)
    assert _rel(o2, o_ref[:, :, T1:]) <= TAU["bf16"]
    assert _rel(S2, S_ref) <= TAU["bf16"]


def test_decode_rejects_bad_arguments(sdl):
    import torch
    d = sdl.make_desc("gdn", "bf16", 1, 1, 2, 128, 128)   # T must be 1
    buf = torch.zeros(1 << 16, dtype=torch.uint8, device="cuda")
    p = buf.data_ptr()
    s = torch.cuda.current_stream().cuda_stream
    assert sdl.dplr_la_decode_step(d, p, p, p, p, p, None, None, None, None, p, p, s) == sdl.dplr.DPLR_ERR_INVALID_ARG
    d = sdl.make_desc("gdn", "bf16", 1, 1, 1, 128, 128)
    assert sdl.dplr_la_decode_step(d, p, p, p, p, p, None, None, None, None, None, p, s) == sdl.dplr.DPLR_ERR_INVALID_ARG
    assert sdl.dplr_la_decode_step(d, p + 4, p, p, p, p, None, None, None, None, p, p, s) == sdl.dplr.DPLR_ERR_INVALID_ARG


@pytest.mark.parametrize("wid", [2, 4])
def test_decode_full_head_count(sdl, wid):
    """The head counts the decode benchmark times (Gated DeltaNet bf16 B8 H16 d128; HDLA bf16 B1 H16 d128): eight
    tokens decoded from a random state for every head, every head against the float64 recurrence."""
    w = workloads.WORKLOADS[wid]
    inp = workloads.generate(w, T=8)
    S0 = (0.1 * np.random.default_rng(9).standard_normal((w.B, w.H, w.dk, w.dv))).astype(np.float32)
    inp["S0"] = S0
    o, S = _decode(sdl, inp, w.mode, w.dtype, S0)
    o_ref, S_ref = oracle.forward_inputs(inp)
    assert _rel(o, o_ref) <= TAU_STEP and _rel(S, S_ref) <= TAU_STEP
