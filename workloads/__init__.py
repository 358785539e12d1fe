"""Seeded synthetic inputs for the chunkwise DPLR-decay linear-attention forward.

This module only draws random inputs with the shapes and value distributions of
the five synthetic workloads. It holds none of the method's arithmetic: no
decay product, no state update, no readout. Both the float64 oracle (test
infrastructure) and the CUDA path are fed from here, so the two share nothing
else.

Recipe (one independent NumPy ``Generator`` per (batch, head), seeded with
``SeedSequence([seed, workload_id, b, h])``; draws in this order per head):

* structured modes (GDN, HDLA): q, k, v ~ N(0, 1) [T, d]; k is l2-normalised per
  token (in float32); then the decay
  Gaussian, then the beta Gaussian.
    - GDN:  decay g_t = logsigmoid(N(0,1))  (one scalar per token, log-space),
            beta_t = sigmoid(N(0,1)).
    - HDLA: decay log(lambda_t) = logsigmoid(N(2,1)) per key channel,
            beta_t = 2 * sigmoid(N(0,1)) in (0, 2).
* generic mode (rank r_ab=4, r_kv=2): q ~ N(0,1); decay log(lambda) =
  logsigmoid(N(2,1)) per channel; beta in (0,2)^4 = 2*sigmoid(N(0,1)) per
  column; U_t = Q factor (reduced QR, NumPy sign convention) of a 64x4
  Gaussian; A_t = Diag(lambda_t) U_t Diag(beta_t), B_t = U_t; K_t, V_t ~
  N(0,1)/8 with two columns each.  Rows of the [T, r, d] arrays are the
  columns of A_t, B_t, K_t, V_t.
* S0 ~ N(0, 0.1^2) per head (standard deviation 0.1) when the workload has a
  nonzero initial state, else absent (zero).

bf16 workloads round q, k, v (and A, B, K, V) to bf16 with round-to-nearest-
even after they are formed in float32; the arrays returned here hold those
rounded values as float32, so upcasting them to bf16 (device) or float64
(oracle) is exact. decay, beta and S0 stay float32 in every workload.
"""

from __future__ import annotations

import concurrent.futures
import dataclasses
import os
from typing import Optional, Sequence

import numpy as np

MODE_GDN = "gdn"
MODE_HDLA = "hdla"
MODE_GENERIC = "generic"


@dataclasses.dataclass(frozen=True)
class Workload:
    wid: int
    name: str
    mode: str
    dtype: str          # "f32" or "bf16": storage type of q/k/v (A/B/K/V)
    B: int
    H: int
    T: int
    dk: int
    dv: int
    r_ab: int
    r_kv: int
    chunk: int
    nonzero_s0: bool

    @property
    def heads(self) -> int:
        return self.B * self.H


WORKLOADS = {
    0: Workload(0, "gdn_f32_b1h2_t256_d32", MODE_GDN, "f32", 1, 2, 256, 32, 32, 1, 1, 64, False),
    1: Workload(1, "hdla_bf16_b4h16_t4096_d128", MODE_HDLA, "bf16", 4, 16, 4096, 128, 128, 2, 1, 64, False),
    2: Workload(2, "gdn_bf16_b8h16_t8192_d128", MODE_GDN, "bf16", 8, 16, 8192, 128, 128, 1, 1, 64, False),
    3: Workload(3, "generic_r4p2_f32_b2h8_t8192_d64", MODE_GENERIC, "f32", 2, 8, 8192, 64, 64, 4, 2, 64, False),
    4: Workload(4, "hdla_bf16_b1h16_t131072_d128_s0", MODE_HDLA, "bf16", 1, 16, 131072, 128, 128, 2, 1, 64, True),
}


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round finite float32 values to the nearest bf16 (ties to even); return float32."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    bits = x.view(np.uint32)
    # finite inputs stay below 2^32 after adding at most 0x8000
    rounded = (bits + np.uint32(0x7FFF) + ((bits >> np.uint32(16)) & np.uint32(1))) & np.uint32(0xFFFF0000)
    return rounded.view(np.float32).reshape(x.shape)


def _logsigmoid(x: np.ndarray) -> np.ndarray:
    return -np.logaddexp(np.float32(0.0), -x)


def _sigmoid(x: np.ndarray) -> np.ndarray:
    return np.float32(0.5) * (np.float32(1.0) + np.tanh(np.float32(0.5) * x))


def _head_rng(seed: int, wid: int, b: int, h: int) -> np.random.Generator:
    return np.random.default_rng(np.random.SeedSequence([seed, wid, b, h]))


def _draw_head(w: Workload, T: int, rng: np.random.Generator) -> dict:
    """Draw one head's inputs (float32 arrays, bf16-rounded where the workload says)."""
    dk, dv = w.dk, w.dv
    f32 = np.float32
    out = {}
    if w.mode in (MODE_GDN, MODE_HDLA):
        q = rng.standard_normal((T, dk), dtype=f32)
        k = rng.standard_normal((T, dk), dtype=f32)
        v = rng.standard_normal((T, dv), dtype=f32)
        nrm = np.sqrt(np.einsum("td,td->t", k, k))
        nrm = np.where(nrm > 0, nrm, np.float32(1.0))
        k = k / nrm[:, None]
        if w.mode == MODE_GDN:
            decay = _logsigmoid(rng.standard_normal(T, dtype=f32))
            beta = _sigmoid(rng.standard_normal(T, dtype=f32))
        else:
            decay = _logsigmoid(rng.standard_normal((T, dk), dtype=f32) + f32(2.0))
            beta = f32(2.0) * _sigmoid(rng.standard_normal(T, dtype=f32))
        if w.dtype == "bf16":
            q, k, v = round_to_bf16(q), round_to_bf16(k), round_to_bf16(v)
        out.update(q=q, k=k, v=v, decay=decay, beta=beta)
    else:
        r, p = w.r_ab, w.r_kv
        q = rng.standard_normal((T, dk), dtype=f32)
        decay = _logsigmoid(rng.standard_normal((T, dk), dtype=f32) + f32(2.0))
        beta = (f32(2.0) * _sigmoid(rng.standard_normal((T, r), dtype=f32))).astype(np.float64)
        g = rng.standard_normal((T, dk, r), dtype=f32).astype(np.float64)
        U, _ = np.linalg.qr(g, mode="reduced")                  # [T, dk, r]
        lam = np.exp(decay.astype(np.float64))                    # [T, dk]
        A = lam[:, :, None] * U * beta[:, None, :]                # D_t U_t diag(beta_t)
        A = np.ascontiguousarray(A.transpose(0, 2, 1)).astype(f32)   # [T, r, dk]
        Bm = np.ascontiguousarray(U.transpose(0, 2, 1)).astype(f32)  # [T, r, dk]
        K = (rng.standard_normal((T, p, dk), dtype=f32) / 8.0).astype(f32)
        V = (rng.standard_normal((T, p, dv), dtype=f32) / 8.0).astype(f32)
        if w.dtype == "bf16":
            q, A, Bm, K, V = (round_to_bf16(x) for x in (q, A, Bm, K, V))
        out.update(q=q, decay=decay, A=A, Bm=Bm, K=K, V=V)
    if w.nonzero_s0:
        out["S0"] = (0.1 * rng.standard_normal((dk, dv), dtype=f32)).astype(f32)
    return out


def generate(w: Workload | int, seed: int = 0, heads: Optional[Sequence[tuple]] = None,
             T: Optional[int] = None) -> dict:
    """Inputs of workload ``w`` in the library layout.

    ``heads``: optional list of (b, h) pairs; the result then has B=1 and
    H=len(heads), each head drawn exactly as in the full workload.
    ``T``: optional shorter sequence; a head's first ``T`` tokens are NOT a
    prefix of the full-length draw (the generator draws whole arrays), so only
    use it for self-contained cases.

    Returns a dict with float32 arrays q/k/v/decay/beta (structured) or
    q/decay/A/Bm/K/V (generic), S0 (or None), plus the workload record and the
    effective B, H, T.
    """
    if isinstance(w, int):
        w = WORKLOADS[w]
    T = w.T if T is None else int(T)
    pairs = [(b, h) for b in range(w.B) for h in range(w.H)] if heads is None else list(heads)
    if heads is None:
        B, H = w.B, w.H
    else:
        B, H = 1, len(pairs)
    first = _draw_head(w, T, _head_rng(seed, w.wid, *pairs[0]))
    res = {key: np.empty((B * H,) + x.shape, dtype=x.dtype) for key, x in first.items()}
    for key, x in first.items():
        res[key][0] = x
    del first

    def fill(i):
        d = _draw_head(w, T, _head_rng(seed, w.wid, *pairs[i]))
        for key, x in d.items():
            res[key][i] = x

    n = len(pairs)
    if n > 1:
        workers = max(1, min(n - 1, os.cpu_count() or 1, 32))
        with concurrent.futures.ThreadPoolExecutor(workers) as pool:
            list(pool.map(fill, range(1, n)))
    for key in list(res):
        res[key] = res[key].reshape((B, H) + res[key].shape[1:])
    for key in ("q", "k", "v", "decay", "beta", "A", "Bm", "K", "V", "S0"):
        res.setdefault(key, None)
    res.update(workload=w, B=B, H=H, T=T)
    return res
