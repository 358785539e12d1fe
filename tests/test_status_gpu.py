"""The device status word through the C ABI, and the fused kernel's timeout path.

Every bounded device-side wait that gives up writes DPLR_ERR_TIMEOUT into the status
word of the workspace, waits for the work its own thread already put in flight
(bulk copies, tensor-core products) and leaves the kernel. The test makes the waits
give up by shrinking their limit with dplr_la_set_wait_limit (no wait is made
endless and nothing is faulted): the call must return, the word must read
DPLR_ERR_TIMEOUT, and the same context must then run a correct forward.
"""

import numpy as np
import pytest

import oracle
import workloads

pytestmark = pytest.mark.gpu

TAU = 2e-2


@pytest.fixture(scope="module")
def sdl():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from structured_decay_linear_gb300 import build as nvbuild
    nvbuild.build()
    import structured_decay_linear_gb300 as s
    s.library()
    yield s
    s.dplr_la_set_wait_limit(0)


def _gdn_case(T, heads=1):
    w = workloads.Workload(95, "gdn_status", "gdn", "bf16", 1, 1, 0, 128, 128, 1, 1, 64, True)
    return w, workloads.generate(w, heads=[(0, h) for h in range(heads)], T=T)


def _dev_args(inp):
    import torch
    d = lambda x, dt: torch.from_numpy(np.ascontiguousarray(x)).to("cuda").to(dt)
    return dict(q=d(inp["q"], torch.bfloat16), k=d(inp["k"], torch.bfloat16), v=d(inp["v"], torch.bfloat16),
                decay=d(inp["decay"], torch.float32), beta=d(inp["beta"], torch.float32),
                S0=d(inp["S0"], torch.float32))


def _rel(a, ref):
    return float(np.abs(a - ref).max() / np.sqrt(np.mean(ref ** 2)))


def test_status_word_reads_zero_after_a_correct_forward(sdl):
    import torch
    w, inp = _gdn_case(200, heads=2)
    f = sdl.Forward("gdn", torch.bfloat16, 1, 2, 200, 128, 128)
    f(**_dev_args(inp))
    assert f.device_status() == sdl.DPLR_OK
    # the two-stage path's workspace starts with a status word as well
    f2 = sdl.Forward("hdla", torch.bfloat16, 1, 1, 64, 64, 64)
    assert f2.device_status() == sdl.DPLR_OK


def test_read_status_rejects_bad_arguments(sdl):
    import torch
    s = torch.cuda.current_stream().cuda_stream
    st, _ = sdl.dplr_la_read_status(None, 256, 0, s)
    assert st == sdl.dplr.DPLR_ERR_WORKSPACE
    buf = torch.zeros(256, dtype=torch.uint8, device="cuda")
    st, _ = sdl.dplr_la_read_status(buf.data_ptr(), 2, 0, s)
    assert st == sdl.dplr.DPLR_ERR_WORKSPACE
    buf[:4].view(torch.int32).fill_(sdl.dplr.DPLR_ERR_TIMEOUT)
    st, word = sdl.dplr_la_read_status(buf.data_ptr(), 256, 1, s)
    assert st == sdl.DPLR_OK and word == sdl.dplr.DPLR_ERR_TIMEOUT
    st, word = sdl.dplr_la_read_status(buf.data_ptr(), 256, 0, s)   # cleared by the previous read
    assert st == sdl.DPLR_OK and word == 0


def test_fused_kernel_timeout_returns_and_reports(sdl):
    """Waits limited to 1000 cycles: the first hand-off between the kernel's warp roles takes
    longer (a chunk's inverse alone is ~3000 cycles), so some wait gives up. The launch must end,
    report DPLR_ERR_TIMEOUT, and the context must stay usable."""
    import torch
    w, inp = _gdn_case(128)
    args = _dev_args(inp)
    f = sdl.Forward("gdn", torch.bfloat16, 1, 1, 128, 128, 128)
    assert f.kernels == 1
    sdl.dplr_la_set_wait_limit(1000)
    try:
        f(**args)                       # a plan made now carries the short limit
        torch.cuda.synchronize()
        assert f.device_status(clear=True) == sdl.dplr.DPLR_ERR_TIMEOUT
    finally:
        sdl.dplr_la_set_wait_limit(0)
    # the same context, default limits: a correct result and a clean status word
    o, ST = f(**args)
    torch.cuda.synchronize()
    assert f.device_status() == sdl.DPLR_OK
    o_ref, S_ref = oracle.forward_inputs(inp)
    assert _rel(o.double().cpu().numpy(), o_ref) <= TAU
    assert _rel(ST.double().cpu().numpy(), S_ref) <= TAU


def test_hdla_tensor_core_kernels_timeout_returns_and_reports(sdl):
    """The same for the tensor-core HDLA stages (chunk maps, then the chain): with every wait limited
    to 1000 cycles the launches end and report DPLR_ERR_TIMEOUT; with the default limit the same
    context gives a correct forward."""
    import torch
    w = workloads.Workload(94, "hdla_status", "hdla", "bf16", 1, 1, 0, 128, 128, 2, 1, 64, True)
    inp = workloads.generate(w, heads=[(0, 0), (0, 1)], T=256)
    args = _dev_args(inp)
    f = sdl.Forward("hdla", torch.bfloat16, 1, 2, 256, 128, 128)
    assert f.path == "hdla_tcgen05"
    sdl.dplr_la_set_wait_limit(1000)
    try:
        f(**args)
        torch.cuda.synchronize()
        assert f.device_status(clear=True) == sdl.dplr.DPLR_ERR_TIMEOUT
    finally:
        sdl.dplr_la_set_wait_limit(0)
    o, ST = f(**args)
    torch.cuda.synchronize()
    assert f.device_status() == sdl.DPLR_OK
    o_ref, S_ref = oracle.forward_inputs(inp)
    assert _rel(o.double().cpu().numpy(), o_ref) <= TAU
    assert _rel(ST.double().cpu().numpy(), S_ref) <= TAU


def test_generic_tensor_core_kernel_timeout_returns_and_reports(sdl):
    """The same for the generic mode's tensor-core chunk kernel (its waits on the tensor cores): limited to 1000
    cycles, the launch ends and reports DPLR_ERR_TIMEOUT; with the default limit the same context is correct."""
    import torch
    from test_parity_gpu import W, gen_generic
    w = W("generic", "f32", 64, 64, 4, 2)
    inp = gen_generic(w, 2, 96, seed=31)
    d = lambda x: torch.from_numpy(np.ascontiguousarray(x)).to("cuda")
    args = dict(q=d(inp["q"]), decay=d(inp["decay"]), A=d(inp["A"]), Bm=d(inp["Bm"]), K=d(inp["K"]), V=d(inp["V"]))
    f = sdl.Forward("generic", torch.float32, 1, 2, 96, 64, 64, r_ab=4, r_kv=2)
    assert f.path == "generic_tcgen05"
    sdl.dplr_la_set_wait_limit(1000)
    try:
        f(**args)
        torch.cuda.synchronize()
        assert f.device_status(clear=True) == sdl.dplr.DPLR_ERR_TIMEOUT
    finally:
        sdl.dplr_la_set_wait_limit(0)
    o, ST = f(**args)
    torch.cuda.synchronize()
    assert f.device_status() == sdl.DPLR_OK
    o_ref, S_ref = oracle.forward_inputs(inp)
    assert _rel(o.double().cpu().numpy(), o_ref) <= 1e-4
    assert _rel(ST.double().cpu().numpy(), S_ref) <= 1e-4
