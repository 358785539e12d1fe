"""Thin ctypes binding of libdplr (argument marshalling only).

Every step of the forward runs in the CUDA kernels of libdplr.so; PyTorch only
provides device memory and the stream. If the library is missing the calls
raise: there is no CPU or PyTorch fallback.
"""

from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional, Tuple

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libdplr.so")

DPLR_OK, DPLR_ERR_INVALID_ARG, DPLR_ERR_UNSUPPORTED, DPLR_ERR_WORKSPACE, DPLR_ERR_CUDA, DPLR_ERR_TIMEOUT = range(6)
DPLR_GDN, DPLR_HDLA, DPLR_GENERIC = 1, 2, 3
DPLR_F32, DPLR_BF16 = 0, 1
MODES = {"gdn": DPLR_GDN, "hdla": DPLR_HDLA, "generic": DPLR_GENERIC}


class dplr_desc(ctypes.Structure):
    _fields_ = [("mode", ctypes.c_int32), ("in_dtype", ctypes.c_int32), ("B", ctypes.c_int32),
                ("H", ctypes.c_int32), ("T", ctypes.c_int32), ("dk", ctypes.c_int32), ("dv", ctypes.c_int32),
                ("r_ab", ctypes.c_int32), ("r_kv", ctypes.c_int32), ("chunk", ctypes.c_int32)]


class DplrError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {status_string(status)}")
        self.status = status


_lock = threading.Lock()
_lib = None
_vp = ctypes.c_void_p


def library() -> ctypes.CDLL:
    """Loads libdplr.so (built in-tree by ``__graft_entry__.build()``)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"{LIB_PATH} is missing: build it first (python -c 'import __graft_entry__ as g; g.build()')")
            lib = ctypes.CDLL(LIB_PATH)
            dp = ctypes.POINTER(dplr_desc)
            lib.dplr_la_workspace_size.restype = ctypes.c_size_t
            lib.dplr_la_workspace_size.argtypes = [dp]
            lib.dplr_la_stage_workspace_size.restype = ctypes.c_size_t
            lib.dplr_la_stage_workspace_size.argtypes = [dp]
            lib.dplr_la_check.restype = ctypes.c_int
            lib.dplr_la_check.argtypes = [dp]
            lib.dplr_la_kernel_count.restype = ctypes.c_int
            lib.dplr_la_kernel_count.argtypes = [dp]
            lib.dplr_status_string.restype = ctypes.c_char_p
            lib.dplr_status_string.argtypes = [ctypes.c_int]
            lib.dplr_la_forward.restype = ctypes.c_int
            lib.dplr_la_forward.argtypes = [dp] + [_vp] * 12 + [_vp, ctypes.c_size_t, _vp]
            lib.dplr_la_chunk_maps.restype = ctypes.c_int
            lib.dplr_la_chunk_maps.argtypes = [dp] + [_vp] * 10 + [_vp, ctypes.c_size_t, _vp]
            lib.dplr_la_state_scan.restype = ctypes.c_int
            lib.dplr_la_state_scan.argtypes = [dp, _vp, _vp, _vp, _vp, ctypes.c_size_t, _vp]
            lib.dplr_la_forward_noalloc.restype = ctypes.c_int
            lib.dplr_la_forward_noalloc.argtypes = [dp] + [_vp] * 12 + [_vp]
            lib.dplr_la_decode_step.restype = ctypes.c_int
            lib.dplr_la_decode_step.argtypes = [dp] + [_vp] * 11 + [_vp]
            lib.dplr_la_backward_workspace_size.restype = ctypes.c_size_t
            lib.dplr_la_backward_workspace_size.argtypes = [dp]
            lib.dplr_la_backward.restype = ctypes.c_int
            lib.dplr_la_backward.argtypes = [dp] + [_vp] * 22 + [_vp, ctypes.c_size_t, _vp]
            lib.dplr_hla_workspace_size.restype = ctypes.c_size_t
            lib.dplr_hla_workspace_size.argtypes = [dp, ctypes.c_int]
            lib.dplr_hla_forward.restype = ctypes.c_int
            lib.dplr_hla_forward.argtypes = [dp] + [_vp] * 6 + [ctypes.c_float, ctypes.c_int, _vp, _vp, ctypes.c_size_t, _vp]
            lib.dplr_hla_path.restype = ctypes.c_char_p
            lib.dplr_hla_path.argtypes = [dp, ctypes.c_int]
            lib.dplr_gdp_workspace_size.restype = ctypes.c_size_t
            lib.dplr_gdp_workspace_size.argtypes = [dp]
            lib.dplr_gdp_forward.restype = ctypes.c_int
            lib.dplr_gdp_forward.argtypes = [dp] + [_vp] * 8 + [_vp, ctypes.c_size_t, _vp]
            lib.dplr_gdp_path.restype = ctypes.c_char_p
            lib.dplr_gdp_path.argtypes = [dp]
            lib.dplr_la_path.restype = ctypes.c_char_p
            lib.dplr_la_path.argtypes = [dp]
            lib.dplr_la_set_wait_limit.restype = None
            lib.dplr_la_set_wait_limit.argtypes = [ctypes.c_longlong]
            lib.dplr_la_read_status.restype = ctypes.c_int
            lib.dplr_la_read_status.argtypes = [_vp, ctypes.c_size_t, ctypes.c_int, ctypes.POINTER(ctypes.c_int), _vp]
            lib.dplr_la_noalloc_status.restype = ctypes.c_int
            lib.dplr_la_noalloc_status.argtypes = [ctypes.POINTER(ctypes.c_int), _vp]
            lib.dplr_la_host_workspace_size.restype = ctypes.c_size_t
            lib.dplr_la_host_workspace_size.argtypes = [dp, ctypes.c_int, ctypes.c_int]
            lib.dplr_la_forward_host.restype = ctypes.c_int
            lib.dplr_la_forward_host.argtypes = [dp] + [_vp] * 12 + [_vp, ctypes.c_size_t, ctypes.c_int,
                                                                     ctypes.c_int, _vp]
            lib.dplr_la_host_seq_workspace_size.restype = ctypes.c_size_t
            lib.dplr_la_host_seq_workspace_size.argtypes = [dp, ctypes.c_int, ctypes.c_int]
            lib.dplr_la_forward_host_seq.restype = ctypes.c_int
            lib.dplr_la_forward_host_seq.argtypes = [dp] + [_vp] * 12 + [_vp, ctypes.c_size_t, ctypes.c_int,
                                                                         ctypes.c_int, _vp]
            _lib = lib
    return _lib


def status_string(status: int) -> str:
    return library().dplr_status_string(int(status)).decode()


def make_desc(mode: str | int, in_dtype, B: int, H: int, T: int, dk: int, dv: int,
              r_ab: Optional[int] = None, r_kv: Optional[int] = None, chunk: int = 64) -> dplr_desc:
    m = MODES[mode] if isinstance(mode, str) else int(mode)
    if in_dtype in (torch.bfloat16, "bf16", DPLR_BF16):
        dt = DPLR_BF16
    elif in_dtype in (torch.float32, "f32", DPLR_F32):
        dt = DPLR_F32
    else:
        raise ValueError(f"unsupported input dtype {in_dtype}")
    if r_ab is None:
        r_ab = {DPLR_GDN: 1, DPLR_HDLA: 2}.get(m, 1)
    if r_kv is None:
        r_kv = 1
    return dplr_desc(m, dt, B, H, T, dk, dv, r_ab, r_kv, chunk)


# ----------------------------------------------------------------------------
# C-ABI mirrors (raw pointers as Python ints, stream as an int handle).
# ----------------------------------------------------------------------------

def dplr_la_workspace_size(desc: dplr_desc) -> int:
    return int(library().dplr_la_workspace_size(ctypes.byref(desc)))


def dplr_la_stage_workspace_size(desc: dplr_desc) -> int:
    return int(library().dplr_la_stage_workspace_size(ctypes.byref(desc)))


def dplr_la_check(desc: dplr_desc) -> int:
    return int(library().dplr_la_check(ctypes.byref(desc)))


def dplr_la_kernel_count(desc: dplr_desc) -> int:
    return int(library().dplr_la_kernel_count(ctypes.byref(desc)))


def dplr_la_decode_step(desc, q, k, v, decay, beta, A, Bm, K, V, S, o, stream) -> int:
    """One recurrent step (desc.T == 1): S updated in place, o = S^T q."""
    return int(library().dplr_la_decode_step(ctypes.byref(desc), q, k, v, decay, beta, A, Bm, K, V, S, o, stream))


def dplr_la_backward_workspace_size(desc: dplr_desc) -> int:
    return int(library().dplr_la_backward_workspace_size(ctypes.byref(desc)))


def dplr_la_backward(desc, q, k, v, decay, beta, A, Bm, K, V, S0, dO, dST, dq, dk, dv, ddecay, dbeta, dA, dBm, dK,
                     dV, dS0, workspace, ws_bytes, stream) -> int:
    """Gradients of every input given dO and dS_T (device pointers; see include/dplr.h)."""
    return int(library().dplr_la_backward(ctypes.byref(desc), q, k, v, decay, beta, A, Bm, K, V, S0, dO, dST, dq, dk,
                                          dv, ddecay, dbeta, dA, dBm, dK, dV, dS0, workspace, ws_bytes, stream))


def dplr_hla_workspace_size(desc: dplr_desc, L: int) -> int:
    return int(library().dplr_hla_workspace_size(ctypes.byref(desc), int(L)))


def dplr_hla_forward(desc, q, k, v, g, beta, W, theta, L, o, workspace, ws_bytes, stream) -> int:
    """HLA's query-gated composition of GDN chunk transitions (device pointers; see include/dplr.h)."""
    return int(library().dplr_hla_forward(ctypes.byref(desc), q, k, v, g, beta, W, float(theta), int(L), o, workspace,
                                          ws_bytes, stream))


def dplr_hla_path(desc, L: int) -> str:
    return library().dplr_hla_path(ctypes.byref(desc), int(L)).decode()


def dplr_gdp_workspace_size(desc: dplr_desc) -> int:
    return int(library().dplr_gdp_workspace_size(ctypes.byref(desc)))


def dplr_gdp_forward(desc, q, k, v, g, beta, S0, o, S_T, workspace, ws_bytes, stream) -> int:
    """Stacked-Householder (Gated DeltaProduct-style) forward (device pointers; see include/dplr.h)."""
    return int(library().dplr_gdp_forward(ctypes.byref(desc), q, k, v, g, beta, S0, o, S_T, workspace, ws_bytes, stream))


def dplr_gdp_path(desc: dplr_desc) -> str:
    return library().dplr_gdp_path(ctypes.byref(desc)).decode()


def dplr_la_path(desc: dplr_desc) -> str:
    return library().dplr_la_path(ctypes.byref(desc)).decode()


def dplr_la_forward(desc, q, k, v, decay, beta, A, Bm, K, V, S0, o, S_T, workspace, ws_bytes, stream) -> int:
    return int(library().dplr_la_forward(ctypes.byref(desc), q, k, v, decay, beta, A, Bm, K, V, S0, o, S_T,
                                         workspace, ctypes.c_size_t(ws_bytes), stream))


def dplr_la_forward_noalloc(desc, q, k, v, decay, beta, A, Bm, K, V, S0, o, S_T, stream) -> int:
    """dplr_la_forward with scratch from the library's fixed device array (no workspace argument)."""
    return int(library().dplr_la_forward_noalloc(ctypes.byref(desc), q, k, v, decay, beta, A, Bm, K, V, S0, o,
                                                 S_T, stream))


def dplr_la_set_wait_limit(cycles: int) -> None:
    """Limit (SM cycles) of the kernels' bounded device-side waits; <= 0 restores the default."""
    library().dplr_la_set_wait_limit(int(cycles))


def dplr_la_read_status(workspace, ws_bytes, clear, stream) -> Tuple[int, int]:
    """Synchronous read of a workspace's device status word: (call status, word)."""
    word = ctypes.c_int(-1)
    st = int(library().dplr_la_read_status(workspace, ctypes.c_size_t(ws_bytes), int(clear), ctypes.byref(word),
                                           stream))
    return st, int(word.value)


def dplr_la_noalloc_status(stream) -> Tuple[int, int]:
    """Synchronous read of the no-alloc scratch array's status word: (call status, word)."""
    word = ctypes.c_int(-1)
    st = int(library().dplr_la_noalloc_status(ctypes.byref(word), stream))
    return st, int(word.value)


def dplr_la_host_workspace_size(desc, groups: int, slots: int) -> int:
    return int(library().dplr_la_host_workspace_size(ctypes.byref(desc), int(groups), int(slots)))


def dplr_la_forward_host(desc, q, k, v, decay, beta, A, Bm, K, V, S0, o, S_T, staging, staging_bytes, groups,
                         slots, stream) -> int:
    """dplr_la_forward with host inputs and outputs; transfers overlapped over groups of heads."""
    return int(library().dplr_la_forward_host(ctypes.byref(desc), q, k, v, decay, beta, A, Bm, K, V, S0, o, S_T,
                                              staging, ctypes.c_size_t(staging_bytes), int(groups), int(slots),
                                              stream))

def dplr_la_host_seq_workspace_size(desc, segments: int, slots: int) -> int:
    return int(library().dplr_la_host_seq_workspace_size(ctypes.byref(desc), int(segments), int(slots)))


def dplr_la_forward_host_seq(desc, q, k, v, decay, beta, A, Bm, K, V, S0, o, S_T, staging, staging_bytes, segments,
                         slots, stream) -> int:
    """dplr_la_forward with host inputs and outputs; transfers overlapped over segments of heads."""
    return int(library().dplr_la_forward_host_seq(ctypes.byref(desc), q, k, v, decay, beta, A, Bm, K, V, S0, o, S_T,
                                              staging, ctypes.c_size_t(staging_bytes), int(segments), int(slots),
                                              stream))


def dplr_la_chunk_maps(desc, q, k, v, decay, beta, A, Bm, K, V, o, workspace, ws_bytes, stream) -> int:
    return int(library().dplr_la_chunk_maps(ctypes.byref(desc), q, k, v, decay, beta, A, Bm, K, V, o,
                                            workspace, ctypes.c_size_t(ws_bytes), stream))


def dplr_la_state_scan(desc, S0, o, S_T, workspace, ws_bytes, stream) -> int:
    return int(library().dplr_la_state_scan(ctypes.byref(desc), S0, o, S_T, workspace,
                                            ctypes.c_size_t(ws_bytes), stream))


# ----------------------------------------------------------------------------
# Tensor-level wrapper.
# ----------------------------------------------------------------------------

def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else t.data_ptr()


def _need(t, name, device, dtype, shape):
    if t is None:
        raise ValueError(f"{name} is required")
    if t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if t.dtype != dtype:
        raise ValueError(f"{name} has dtype {t.dtype}, expected {dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


class Forward:
    """Prepared forward for one descriptor: owns the output and workspace tensors so that
    repeated calls (benchmarks, CUDA graphs) allocate nothing."""

    def __init__(self, mode: str, in_dtype: torch.dtype, B: int, H: int, T: int, dk: int, dv: int,
                 r_ab: Optional[int] = None, r_kv: Optional[int] = None, chunk: int = 64,
                 device: Optional[torch.device] = None):
        self.desc = make_desc(mode, in_dtype, B, H, T, dk, dv, r_ab, r_kv, chunk)
        st = dplr_la_check(self.desc)
        if st != DPLR_OK:
            raise DplrError(st, "dplr_la_check")
        self.mode, self.in_dtype = MODES[mode] if isinstance(mode, str) else mode, in_dtype
        self.B, self.H, self.T, self.dk, self.dv = B, H, T, dk, dv
        self.r_ab, self.r_kv = self.desc.r_ab, self.desc.r_kv
        self.device = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
        self.ws_bytes = dplr_la_workspace_size(self.desc)
        # zeroed once: on the fused path its first int32 is the device status word
        self.workspace = torch.zeros(max(self.ws_bytes, 256), dtype=torch.uint8, device=self.device)
        self.stage_ws_bytes = dplr_la_stage_workspace_size(self.desc)
        self._stage_ws = None
        self.o = torch.empty((B, H, T, dv), dtype=torch.float32, device=self.device)
        self.S_T = torch.empty((B, H, dk, dv), dtype=torch.float32, device=self.device)
        self.kernels = dplr_la_kernel_count(self.desc)
        self.path = dplr_la_path(self.desc)

    def _check(self, q, k, v, decay, beta, A, Bm, K, V, S0):
        B, H, T, dk, dv, dev, dt = self.B, self.H, self.T, self.dk, self.dv, self.device, self.in_dtype
        _need(q, "q", dev, dt, (B, H, T, dk))
        if self.mode == DPLR_GENERIC:
            _need(decay, "decay", dev, torch.float32, (B, H, T, dk))
            _need(A, "A", dev, dt, (B, H, T, self.r_ab, dk))
            _need(Bm, "Bm", dev, dt, (B, H, T, self.r_ab, dk))
            if self.r_kv > 0:
                _need(K, "K", dev, dt, (B, H, T, self.r_kv, dk))
                _need(V, "V", dev, dt, (B, H, T, self.r_kv, dv))
        else:
            _need(k, "k", dev, dt, (B, H, T, dk))
            _need(v, "v", dev, dt, (B, H, T, dv))
            _need(decay, "decay", dev, torch.float32, (B, H, T) if self.mode == DPLR_GDN else (B, H, T, dk))
            _need(beta, "beta", dev, torch.float32, (B, H, T))
        if S0 is not None:
            _need(S0, "S0", dev, torch.float32, (B, H, dk, dv))

    def __call__(self, q, k=None, v=None, decay=None, beta=None, A=None, Bm=None, K=None, V=None, S0=None,
                 stream: Optional[torch.cuda.Stream] = None, check: bool = True) -> Tuple[torch.Tensor, torch.Tensor]:
        if check:
            self._check(q, k, v, decay, beta, A, Bm, K, V, S0)
        s = stream if stream is not None else torch.cuda.current_stream(self.device)
        st = dplr_la_forward(self.desc, _ptr(q), _ptr(k), _ptr(v), _ptr(decay), _ptr(beta), _ptr(A), _ptr(Bm),
                             _ptr(K), _ptr(V), _ptr(S0), _ptr(self.o), _ptr(self.S_T), _ptr(self.workspace),
                             self.ws_bytes, s.cuda_stream)
        if st != DPLR_OK:
            raise DplrError(st, "dplr_la_forward")
        return self.o, self.S_T

    def device_status(self, clear: bool = False) -> int:
        """The workspace's device status word (0, or DPLR_ERR_TIMEOUT after a bounded wait gave up),
        read synchronously through dplr_la_read_status."""
        s = torch.cuda.current_stream(self.device)
        st, word = dplr_la_read_status(_ptr(self.workspace), self.workspace.numel(), clear, s.cuda_stream)
        if st != DPLR_OK:
            raise DplrError(st, "dplr_la_read_status")
        return word

    def _stage_workspace(self):
        if self._stage_ws is None:
            self._stage_ws = torch.empty(max(self.stage_ws_bytes, 256), dtype=torch.uint8, device=self.device)
        return self._stage_ws

    def chunk_maps(self, q, k=None, v=None, decay=None, beta=None, A=None, Bm=None, K=None, V=None,
                   stream: Optional[torch.cuda.Stream] = None):
        s = stream if stream is not None else torch.cuda.current_stream(self.device)
        st = dplr_la_chunk_maps(self.desc, _ptr(q), _ptr(k), _ptr(v), _ptr(decay), _ptr(beta), _ptr(A), _ptr(Bm),
                                _ptr(K), _ptr(V), _ptr(self.o), _ptr(self._stage_workspace()), self.stage_ws_bytes,
                                s.cuda_stream)
        if st != DPLR_OK:
            raise DplrError(st, "dplr_la_chunk_maps")

    def state_scan(self, S0=None, stream: Optional[torch.cuda.Stream] = None):
        s = stream if stream is not None else torch.cuda.current_stream(self.device)
        st = dplr_la_state_scan(self.desc, _ptr(S0), _ptr(self.o), _ptr(self.S_T), _ptr(self._stage_workspace()),
                                self.stage_ws_bytes, s.cuda_stream)
        if st != DPLR_OK:
            raise DplrError(st, "dplr_la_state_scan")
        return self.o, self.S_T


def default_groups(desc: dplr_desc) -> int:
    """Head groups for dplr_la_forward_host: enough groups to overlap the copies, while each
    group keeps enough heads to occupy the GPU (the fused kernel runs one CTA per head for the
    whole sequence, the two-stage kernels parallelise over chunks and want more heads)."""
    bh = desc.B * desc.H
    min_heads = 16 if dplr_la_kernel_count(desc) == 1 else 32
    best = 1
    for g in range(1, 17):
        if bh % g == 0 and bh // g >= min_heads:
            best = g
    return best


class ForwardHost:
    """Prepared forward from host (pinned) tensors through dplr_la_forward_host: owns the device
    staging area and pinned host outputs, so repeated calls allocate nothing."""

    def __init__(self, mode: str, in_dtype: torch.dtype, B: int, H: int, T: int, dk: int, dv: int,
                 r_ab: Optional[int] = None, r_kv: Optional[int] = None, chunk: int = 64,
                 groups: Optional[int] = None, slots: int = 8, device: Optional[torch.device] = None):
        self.desc = make_desc(mode, in_dtype, B, H, T, dk, dv, r_ab, r_kv, chunk)
        st = dplr_la_check(self.desc)
        if st != DPLR_OK:
            raise DplrError(st, "dplr_la_check")
        self.groups = groups if groups is not None else default_groups(self.desc)
        self.slots = slots
        self.device = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
        self.staging_bytes = dplr_la_host_workspace_size(self.desc, self.groups, self.slots)
        if self.staging_bytes == 0:
            raise DplrError(DPLR_ERR_INVALID_ARG, "dplr_la_host_workspace_size")
        self.staging = torch.empty(self.staging_bytes, dtype=torch.uint8, device=self.device)
        self.o = torch.empty((B, H, T, dv), dtype=torch.float32).pin_memory()
        self.S_T = torch.empty((B, H, dk, dv), dtype=torch.float32).pin_memory()

    def __call__(self, q, k=None, v=None, decay=None, beta=None, A=None, Bm=None, K=None, V=None, S0=None,
                 stream: Optional[torch.cuda.Stream] = None) -> Tuple[torch.Tensor, torch.Tensor]:
        """Host tensors in, host tensors out (valid once `stream` has been synchronised)."""
        for name, t in (("q", q), ("k", k), ("v", v), ("decay", decay), ("beta", beta), ("A", A), ("Bm", Bm),
                        ("K", K), ("V", V), ("S0", S0)):
            if t is not None and (t.device.type != "cpu" or not t.is_contiguous()):
                raise ValueError(f"{name} must be a contiguous host tensor")
        s = stream if stream is not None else torch.cuda.current_stream(self.device)
        st = dplr_la_forward_host(self.desc, _ptr(q), _ptr(k), _ptr(v), _ptr(decay), _ptr(beta), _ptr(A), _ptr(Bm),
                                  _ptr(K), _ptr(V), _ptr(S0), _ptr(self.o), _ptr(self.S_T), _ptr(self.staging),
                                  self.staging_bytes, self.groups, self.slots, s.cuda_stream)
        if st != DPLR_OK:
            raise DplrError(st, "dplr_la_forward_host")
        return self.o, self.S_T


def default_segments(T: int) -> int:
    """Sequence segments for dplr_la_forward_host_seq: 4 up to 32K tokens, then one per 8K tokens (at most 16).
    Shorter segments shorten the tail after the last copy in, but each head's row of a 2-D copy shrinks
    with them, and rows well under ~0.5 MB copy slowly."""
    return 4 if T < 32768 else max(4, min(16, T // 8192))


class ForwardHostSeq:
    """Prepared forward from host (pinned) tensors through dplr_la_forward_host_seq (the sequence split
    into segments whose forwards carry the state on the device): owns the device staging area and pinned
    host outputs, so repeated calls allocate nothing."""

    def __init__(self, mode: str, in_dtype: torch.dtype, B: int, H: int, T: int, dk: int, dv: int,
                 r_ab: Optional[int] = None, r_kv: Optional[int] = None, chunk: int = 64,
                 segments: Optional[int] = None, slots: int = 4, device: Optional[torch.device] = None):
        self.desc = make_desc(mode, in_dtype, B, H, T, dk, dv, r_ab, r_kv, chunk)
        st = dplr_la_check(self.desc)
        if st != DPLR_OK:
            raise DplrError(st, "dplr_la_check")
        self.segments = segments if segments is not None else default_segments(T)
        self.slots = slots
        self.device = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
        self.staging_bytes = dplr_la_host_seq_workspace_size(self.desc, self.segments, self.slots)
        if self.staging_bytes == 0:
            raise DplrError(DPLR_ERR_INVALID_ARG, "dplr_la_host_seq_workspace_size")
        self.staging = torch.empty(self.staging_bytes, dtype=torch.uint8, device=self.device)
        self.o = torch.empty((B, H, T, dv), dtype=torch.float32).pin_memory()
        self.S_T = torch.empty((B, H, dk, dv), dtype=torch.float32).pin_memory()

    def __call__(self, q, k=None, v=None, decay=None, beta=None, A=None, Bm=None, K=None, V=None, S0=None,
                 stream: Optional[torch.cuda.Stream] = None) -> Tuple[torch.Tensor, torch.Tensor]:
        """Host tensors in, host tensors out (valid once `stream` has been synchronised)."""
        for name, t in (("q", q), ("k", k), ("v", v), ("decay", decay), ("beta", beta), ("A", A), ("Bm", Bm),
                        ("K", K), ("V", V), ("S0", S0)):
            if t is not None and (t.device.type != "cpu" or not t.is_contiguous()):
                raise ValueError(f"{name} must be a contiguous host tensor")
        s = stream if stream is not None else torch.cuda.current_stream(self.device)
        st = dplr_la_forward_host_seq(self.desc, _ptr(q), _ptr(k), _ptr(v), _ptr(decay), _ptr(beta), _ptr(A),
                                      _ptr(Bm), _ptr(K), _ptr(V), _ptr(S0), _ptr(self.o), _ptr(self.S_T),
                                      _ptr(self.staging), self.staging_bytes, self.segments, self.slots,
                                      s.cuda_stream)
        if st != DPLR_OK:
            raise DplrError(st, "dplr_la_forward_host_seq")
        return self.o, self.S_T


def forward(mode: str, q, k=None, v=None, decay=None, beta=None, A=None, Bm=None, K=None, V=None, S0=None,
            chunk: int = 64) -> Tuple[torch.Tensor, torch.Tensor]:
    """One-shot forward on device tensors; returns fresh (o [B,H,T,dv] fp32, S_T [B,H,dk,dv] fp32)."""
    B, H, T, dk = q.shape
    if mode == "generic":
        r_ab, r_kv = A.shape[3], (K.shape[3] if K is not None else 0)
        dv = V.shape[4] if V is not None else S0.shape[3]
    else:
        r_ab, r_kv, dv = None, None, v.shape[3]
    f = Forward(mode, q.dtype, B, H, T, dk, dv, r_ab, r_kv, chunk, device=q.device)
    return f(q, k, v, decay, beta, A, Bm, K, V, S0)


class Decode:
    """Prepared one-token step for B x H heads (dplr_la_decode_step): owns the state S and the output o."""

    def __init__(self, mode: str, in_dtype: torch.dtype, B: int, H: int, dk: int, dv: int,
                 r_ab: Optional[int] = None, r_kv: Optional[int] = None, S0: Optional[torch.Tensor] = None,
                 device: Optional[torch.device] = None):
        self.desc = make_desc(mode, in_dtype, B, H, 1, dk, dv, r_ab, r_kv)
        st = dplr_la_check(self.desc)
        if st != DPLR_OK:
            raise DplrError(st, "dplr_la_check")
        self.device = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
        self.S = torch.zeros((B, H, dk, dv), dtype=torch.float32, device=self.device)
        if S0 is not None:
            self.S.copy_(S0)
        self.o = torch.empty((B, H, 1, dv), dtype=torch.float32, device=self.device)

    def __call__(self, q, k=None, v=None, decay=None, beta=None, A=None, Bm=None, K=None, V=None,
                 stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
        """One token (tensors with T = 1, contiguous, on the device). Returns o [B,H,1,dv]."""
        s = stream if stream is not None else torch.cuda.current_stream(self.device)
        st = dplr_la_decode_step(self.desc, _ptr(q), _ptr(k), _ptr(v), _ptr(decay), _ptr(beta), _ptr(A), _ptr(Bm),
                                 _ptr(K), _ptr(V), _ptr(self.S), _ptr(self.o), s.cuda_stream)
        if st != DPLR_OK:
            raise DplrError(st, "dplr_la_decode_step")
        return self.o


class Backward:
    """Prepared backward for one descriptor (dplr_la_backward): owns the workspace and the fp32 gradients."""

    def __init__(self, mode: str, in_dtype: torch.dtype, B: int, H: int, T: int, dk: int, dv: int,
                 r_ab: Optional[int] = None, r_kv: Optional[int] = None, chunk: int = 64,
                 device: Optional[torch.device] = None):
        self.mode = mode
        self.desc = make_desc(mode, in_dtype, B, H, T, dk, dv, r_ab, r_kv, chunk)
        self.device = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
        nbytes = dplr_la_backward_workspace_size(self.desc)
        if nbytes == 0:
            raise DplrError(dplr_la_check(self.desc) or 2, "dplr_la_backward_workspace_size")
        self.ws = torch.empty(nbytes + 256, dtype=torch.uint8, device=self.device)
        off = (-self.ws.data_ptr()) % 256
        self.ws_ptr, self.ws_bytes = self.ws.data_ptr() + off, nbytes
        r, p = self.desc.r_ab, self.desc.r_kv
        f = lambda *shape: torch.zeros(shape, dtype=torch.float32, device=self.device)
        g = {"q": f(B, H, T, dk), "S0": f(B, H, dk, dv)}
        if mode == "generic":
            g.update(decay=f(B, H, T, dk), A=f(B, H, T, r, dk), Bm=f(B, H, T, r, dk))
            if p > 0:
                g.update(K=f(B, H, T, p, dk), V=f(B, H, T, p, dv))
        else:
            g.update(k=f(B, H, T, dk), v=f(B, H, T, dv), beta=f(B, H, T),
                     decay=f(B, H, T) if mode == "gdn" else f(B, H, T, dk))
        self.grads = g

    def __call__(self, dO, dST=None, q=None, k=None, v=None, decay=None, beta=None, A=None, Bm=None, K=None,
                 V=None, S0=None, stream: Optional[torch.cuda.Stream] = None) -> dict:
        """Gradients of the forward's inputs (dict of fp32 tensors, also kept in .grads)."""
        s = stream if stream is not None else torch.cuda.current_stream(self.device)
        g = self.grads
        st = dplr_la_backward(self.desc, _ptr(q), _ptr(k), _ptr(v), _ptr(decay), _ptr(beta), _ptr(A), _ptr(Bm),
                              _ptr(K), _ptr(V), _ptr(S0), _ptr(dO), _ptr(dST), _ptr(g["q"]), _ptr(g.get("k")),
                              _ptr(g.get("v")), _ptr(g["decay"]), _ptr(g.get("beta")), _ptr(g.get("A")),
                              _ptr(g.get("Bm")), _ptr(g.get("K")), _ptr(g.get("V")), _ptr(g["S0"]), self.ws_ptr,
                              self.ws_bytes, s.cuda_stream)
        if st != DPLR_OK:
            raise DplrError(st, "dplr_la_backward")
        return g


class HLA:
    """Prepared HLA forward (dplr_hla_forward) for one GDN descriptor and chunk length: owns workspace and output."""

    def __init__(self, in_dtype: torch.dtype, B: int, H: int, T: int, dk: int, dv: int, L: int = 256,
                 device: Optional[torch.device] = None):
        self.desc = make_desc("gdn", in_dtype, B, H, T, dk, dv)
        self.L = int(L)
        self.device = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
        nbytes = dplr_hla_workspace_size(self.desc, self.L)
        if nbytes == 0:
            raise DplrError(2, "dplr_hla_workspace_size")
        self.ws = torch.empty(nbytes + 256, dtype=torch.uint8, device=self.device)
        off = (-self.ws.data_ptr()) % 256
        self.ws_ptr, self.ws_bytes = self.ws.data_ptr() + off, nbytes
        self.o = torch.empty((B, H, T, dv), dtype=torch.float32, device=self.device)
        self.path = dplr_hla_path(self.desc, self.L)

    def device_status(self, clear: bool = False) -> int:
        """The workspace's status word (0, or DPLR_ERR_TIMEOUT after a bounded wait gave up), read synchronously."""
        s = torch.cuda.current_stream(self.device)
        st, word = dplr_la_read_status(self.ws_ptr, self.ws_bytes, clear, s.cuda_stream)
        if st != DPLR_OK:
            raise DplrError(st, "dplr_la_read_status")
        return word

    def __call__(self, q, k, v, g, beta, W, theta: float = 0.0,
                 stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
        s = stream if stream is not None else torch.cuda.current_stream(self.device)
        st = dplr_hla_forward(self.desc, _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(W), theta, self.L,
                              _ptr(self.o), self.ws_ptr, self.ws_bytes, s.cuda_stream)
        if st != DPLR_OK:
            raise DplrError(st, "dplr_hla_forward")
        return self.o


class GDP:
    """Prepared stacked-Householder forward (dplr_gdp_forward) with n_h steps per token: owns workspace and outputs."""

    def __init__(self, in_dtype: torch.dtype, B: int, H: int, T: int, dk: int, dv: int, nh: int,
                 device: Optional[torch.device] = None):
        self.desc = make_desc("generic", in_dtype, B, H, T, dk, dv, nh, nh)
        self.device = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
        nbytes = dplr_gdp_workspace_size(self.desc)
        if nbytes == 0:
            raise DplrError(2, "dplr_gdp_workspace_size")
        self.ws = torch.empty(nbytes + 256, dtype=torch.uint8, device=self.device)
        off = (-self.ws.data_ptr()) % 256
        self.ws_ptr, self.ws_bytes = self.ws.data_ptr() + off, nbytes
        self.o = torch.empty((B, H, T, dv), dtype=torch.float32, device=self.device)
        self.S_T = torch.empty((B, H, dk, dv), dtype=torch.float32, device=self.device)
        self.path = dplr_gdp_path(self.desc)

    def __call__(self, q, k, v, g, beta, S0=None, stream: Optional[torch.cuda.Stream] = None):
        s = stream if stream is not None else torch.cuda.current_stream(self.device)
        st = dplr_gdp_forward(self.desc, _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(S0), _ptr(self.o),
                              _ptr(self.S_T), self.ws_ptr, self.ws_bytes, s.cuda_stream)
        if st != DPLR_OK:
            raise DplrError(st, "dplr_gdp_forward")
        return self.o, self.S_T
