"""The forward and the decode step replayed from a CUDA graph.

The prepared bindings (Forward, Decode) own their outputs and workspace, so a call allocates nothing and can be
captured once and replayed: the replay must give the same bits as a direct call on the same inputs, also after
the inputs are changed in place between replays (the graph reads them through the same pointers).
"""

import pytest

pytestmark = pytest.mark.gpu


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


def _inputs(mode, dt, B, H, T, d, r=None, p=None, seed=0):
    import torch
    g = torch.Generator(device="cuda").manual_seed(seed)
    rn = lambda *s: torch.randn(*s, device="cuda", generator=g)
    x = {"q": (rn(B, H, T, d) / d ** 0.5).to(dt)}
    if mode == "generic":   # P_t = Diag(lambda) (I - U Diag(beta) U^T), U orthonormal, beta in (0, 2): stable
        lam = torch.sigmoid(2 + rn(B, H, T, d))
        U = torch.linalg.qr(rn(B, H, T, d, r)).Q                      # [B,H,T,d,r]
        bet = 2 * torch.sigmoid(rn(B, H, T, r))
        x["decay"] = torch.log(lam)
        x["A"] = (lam.unsqueeze(-1) * U * bet.unsqueeze(-2)).transpose(-1, -2).contiguous().to(dt)
        x["Bm"] = U.transpose(-1, -2).contiguous().to(dt)
        x["K"] = (rn(B, H, T, p, d) / 8).to(dt)
        x["V"] = (rn(B, H, T, p, d) / 8).to(dt)
    else:
        x["k"] = torch.nn.functional.normalize(rn(B, H, T, d), dim=-1).to(dt)
        x["v"] = rn(B, H, T, d).to(dt)
        x["decay"] = (torch.nn.functional.logsigmoid(rn(B, H, T)) if mode == "gdn"
                      else torch.nn.functional.logsigmoid(2 + rn(B, H, T, d)))
        x["beta"] = torch.sigmoid(rn(B, H, T)) * (2.0 if mode == "hdla" else 1.0)
    return x


CASES = [
    # mode, dtype, B, H, T, d, r, p   (the fused kernel; the tensor-core HDLA and generic stages; the fp32 stages)
    ("gdn", "bf16", 1, 4, 1000, 128, None, None),
    ("hdla", "bf16", 1, 4, 1000, 128, None, None),
    ("generic", "f32", 1, 2, 600, 64, 4, 2),
    ("gdn", "f32", 2, 2, 300, 32, None, None),
]


@pytest.mark.parametrize("mode,dtype,B,H,T,d,r,p", CASES)
def test_forward_replays_from_a_graph(sdl, mode, dtype, B, H, T, d, r, p):
    import torch
    dt = torch.bfloat16 if dtype == "bf16" else torch.float32
    x = _inputs(mode, dt, B, H, T, d, r, p)
    S0 = 0.1 * torch.randn(B, H, d, d, device="cuda")
    f = sdl.Forward(mode, dt, B, H, T, d, d, r, p)
    o, S_T = f(**x, S0=S0)            # direct call (also the warm-up: per-device settings happen here)
    o_ref, S_ref = o.clone(), S_T.clone()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        f(**x, S0=S0, check=False)
    f.o.zero_()
    f.S_T.zero_()
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(f.o, o_ref) and torch.equal(f.S_T, S_ref)
    # new values in the same buffers: the replay reads them
    for key in x:
        x[key].mul_(0.5 if key != "decay" else 1.0)
    S0.mul_(-1.0)
    graph.replay()
    torch.cuda.synchronize()
    o_g, S_g = f.o.clone(), f.S_T.clone()
    o_d, S_d = f(**x, S0=S0)
    torch.cuda.synchronize()
    assert torch.equal(o_g, o_d) and torch.equal(S_g, S_d)
    assert not torch.equal(o_g, o_ref)
    assert f.device_status() == 0


@pytest.mark.parametrize("mode", ["gdn", "hdla"])
def test_decode_steps_replay_from_a_graph(sdl, mode):
    """Twenty decode steps captured as one graph equal twenty direct steps from the same state."""
    import torch
    B, H, d, n = 2, 3, 128, 20
    x = _inputs(mode, torch.bfloat16, B, H, n, d, seed=1)
    tok = [{k_: v_[:, :, t:t + 1].contiguous() for k_, v_ in x.items()} for t in range(n)]
    S0 = 0.1 * torch.randn(B, H, d, d, device="cuda")
    direct = sdl.Decode(mode, torch.bfloat16, B, H, d, d, S0=S0)
    outs = [direct(**tok[t]).clone() for t in range(n)]
    step = sdl.Decode(mode, torch.bfloat16, B, H, d, d, S0=S0)
    step(**tok[0])                    # warm-up, then the state is reset
    step.S.copy_(S0)
    torch.cuda.synchronize()
    captured = torch.empty(n, B, H, 1, d, device="cuda")
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for t in range(n):
            captured[t].copy_(step(**tok[t]))
    step.S.copy_(S0)
    graph.replay()
    torch.cuda.synchronize()
    for t in range(n):
        assert torch.equal(captured[t], outs[t]), t
    assert torch.equal(step.S, direct.S)
