"""The allocation-free forward (dplr_la_forward_noalloc) against the regular entry point.

Callers that cannot allocate device memory at call time (an engine that reserved the
device up front, a plugin whose host framework owns the allocator) use this entry point:
it takes its scratch from a fixed array inside the library. This file is collected last
so that a failure here leaves every other test already run.
"""

import numpy as np
import pytest

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


def _dev(x, dtype):
    import torch
    return None if x is None else torch.from_numpy(np.ascontiguousarray(x)).to("cuda").to(dtype)


def _case(w, heads, T):
    import torch
    inp = workloads.generate(w, heads=[(0, h) for h in range(heads)], T=T)
    dt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    args = dict(q=_dev(inp["q"], dt), k=_dev(inp["k"], dt), v=_dev(inp["v"], dt),
                decay=_dev(inp["decay"], torch.float32), beta=_dev(inp["beta"], torch.float32),
                A=None, Bm=None, K=None, V=None, S0=_dev(inp["S0"], torch.float32))
    return inp, dt, args


def _noalloc(sdl, desc, args, o, ST):
    import torch
    p = lambda t: None if t is None else t.data_ptr()
    st = sdl.dplr_la_forward_noalloc(desc, p(args["q"]), p(args["k"]), p(args["v"]), p(args["decay"]),
                                     p(args["beta"]), None, None, None, None, p(args["S0"]), o.data_ptr(),
                                     ST.data_ptr(), torch.cuda.current_stream().cuda_stream)
    return st


def _rel(a, b):
    a, b = a.double().cpu().numpy(), b.double().cpu().numpy()
    return float(np.abs(a - b).max() / max(np.sqrt(np.mean(b ** 2)), 1e-30))


def test_noalloc_matches_forward_on_two_calls_in_a_row(sdl):
    import torch
    cases = [
        workloads.Workload(98, "hdla_noalloc", "hdla", "bf16", 1, 1, 0, 128, 128, 2, 1, 64, True),
        workloads.Workload(97, "gdn_noalloc", "gdn", "f32", 1, 1, 0, 64, 32, 1, 1, 64, True),
        # GDN bf16 d=128 runs the fused kernel: its scratch is the status word
        workloads.Workload(96, "gdn_fused_noalloc", "gdn", "bf16", 1, 1, 0, 128, 128, 1, 1, 64, True),
    ]
    for w, heads, T in ((cases[0], 3, 300), (cases[1], 2, 130), (cases[2], 3, 257)):
        inp, dt, args = _case(w, heads, T)
        ref = sdl.Forward(w.mode, dt, 1, heads, T, w.dk, w.dv)
        o_ref, S_ref = [x.clone() for x in ref(**args)]
        for call in range(2):   # two calls in a row reuse the same scratch array
            o = torch.full_like(o_ref, float("nan"))
            ST = torch.full_like(S_ref, float("nan"))
            torch.cuda.synchronize()
            free_before = torch.cuda.mem_get_info()[0]
            assert _noalloc(sdl, ref.desc, args, o, ST) == sdl.DPLR_OK
            torch.cuda.synchronize()
            if call == 1:   # the array is reserved by the first call on the device; later calls take nothing
                assert torch.cuda.mem_get_info()[0] == free_before
            st, word = sdl.dplr_la_noalloc_status(torch.cuda.current_stream().cuda_stream)
            assert st == sdl.DPLR_OK and word == sdl.DPLR_OK
            assert _rel(o, o_ref) <= TAU[w.dtype]
            assert _rel(ST, S_ref) <= TAU[w.dtype]


def test_noalloc_rejects_problems_beyond_its_scratch(sdl):
    import torch
    d = sdl.make_desc("hdla", "bf16", 4, 16, 4096, 128, 128)
    assert sdl.dplr_la_workspace_size(d) > 64 * 2 ** 20
    fake = 1 << 20    # never dereferenced: the size check comes first
    st = sdl.dplr_la_forward_noalloc(d, fake, fake, fake, fake, fake, None, None, None, None, None, fake, None,
                                     torch.cuda.current_stream().cuda_stream)
    assert st == sdl.dplr.DPLR_ERR_UNSUPPORTED
