"""Helpers shared by the GPU parity tests: moving generated inputs to the
device and comparing against the oracle."""
from __future__ import annotations

import numpy as np
import torch

import workloads as W

# parity bars: relative L2 of o and h_final, max-abs on L2-normalised q/k
TOL_REL_L2 = {"bf16": 1e-2, "f32": 1e-4}
TOL_MAX_ABS = 2e-2


def dev():
    return torch.device("cuda", 0)


def to_dev(a: np.ndarray, dtype: str):
    """Generated array (bf16 bits or fp32) -> CUDA tensor of that dtype."""
    if dtype == "bf16":
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev())
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(dev())


def f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def rel_l2(a, b) -> float:
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    nb = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / (nb if nb > 0 else 1.0))


def assert_close(got, exp, dtype: str, what: str, max_abs=True):
    r = rel_l2(got, exp)
    assert r <= TOL_REL_L2[dtype], f"{what}: relative L2 {r:.3e} > {TOL_REL_L2[dtype]}"
    if max_abs:
        m = float(np.max(np.abs(np.asarray(got, np.float64) - np.asarray(exp, np.float64)))) \
            if np.size(exp) else 0.0
        assert m <= TOL_MAX_ABS, f"{what}: max abs error {m:.3e} > {TOL_MAX_ABS}"
    return r


def chunk_inputs(w: W.Workload):
    """Generated q/k/v/g/beta/h0 of a workload as (numpy, device) pairs."""
    q, k, v, g, b = w.q(), w.k(), w.v(), w.g(), w.beta()
    h0 = w.h0()
    host = dict(q=W.as_f64(q, w.dtype).reshape(w.T, w.Hk, w.dk),
                k=W.as_f64(k, w.dtype).reshape(w.T, w.Hk, w.dk),
                v=W.as_f64(v, w.dtype).reshape(w.T, w.Hv, w.dv),
                g=g.astype(np.float64), beta=W.as_f64(b, w.dtype),
                h0=None if h0 is None else h0.astype(np.float64))
    d = dict(q=to_dev(q, w.dtype).view(w.T, w.Hk, w.dk),
             k=to_dev(k, w.dtype).view(w.T, w.Hk, w.dk),
             v=to_dev(v, w.dtype).view(w.T, w.Hv, w.dv),
             g=to_dev(g, "f32"), beta=to_dev(b, w.dtype),
             h0=None if h0 is None else to_dev(h0, "f32"),
             cu=torch.from_numpy(w.cu_seqlens()).to(dev()))
    return host, d


def path_inputs(w: W.Workload):
    """Generated raw conv input, conv weights and gates as (numpy, device)."""
    x, cw, cb, g, b = w.x(), w.conv_w(), w.conv_b(), w.g(), w.beta()
    h0 = w.h0()
    host = dict(x=x, conv_w=W.as_f64(cw, w.dtype), conv_b=None if cb is None else W.as_f64(cb, w.dtype),
                g=g.astype(np.float64), beta=W.as_f64(b, w.dtype),
                h0=None if h0 is None else h0.astype(np.float64))
    d = dict(x=to_dev(x, w.dtype), conv_w=to_dev(cw, w.dtype),
             conv_b=None if cb is None else to_dev(cb, w.dtype),
             g=to_dev(g, "f32"), beta=to_dev(b, w.dtype),
             h0=None if h0 is None else to_dev(h0, "f32"),
             cu=torch.from_numpy(w.cu_seqlens()).to(dev()))
    return host, d
