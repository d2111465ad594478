"""fp64 CPU oracle for the context-parallel Gated DeltaNet forward.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
bench's CPU-baseline leg are the only callers.  The CUDA library never
imports, links or runs anything here, and this package shares no code with
it.  The arithmetic lives in ``gdn_oracle.c`` (plain loops, fp64, the
defining formulas of the source pages written out); this file only marshals
numpy arrays into it.

Sources: flash-linear-attention ``fla/ops/cp/context.py``
(``get_cp_cu_seqlens``, steps 1-5) for the shard plan; hyper-parallel
``linear_attention_context_parallel.py`` (``_causal_conv1d_with_cp_halo``,
``_l2norm_torch``, the chunked gated delta rule, the state summary and the
prefix merge) for everything else; the backward (``gdn_backward``) is the
reverse-mode gradient of the token recurrence, whose state gradient flows
the way the page's ``_RecvInitialStateP2PFunction`` /
``_SendFinalStateP2PFunction`` send it back.

Every function here is pinned by ``tests/test_oracle_pins.py`` against
brute force, closed forms, library routines or an independent restatement.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdn_oracle.c")
_SO = os.path.join(_HERE, "_gdn_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle into a host shared library next to its source."""
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".{os.getpid()}.tmp"
        subprocess.run(["gcc", "-O2", "-ffp-contract=off", "-fopenmp", "-fPIC", "-shared",
                        "-o", tmp, _SRC, "-lm"], check=True)
        os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i64, dbl, vp, i32 = ctypes.c_int64, ctypes.c_double, ctypes.c_void_p, ctypes.c_int
            lib.orc_plan_shard.argtypes = [vp, i64, i64, i64, vp, vp, vp]
            lib.orc_plan_shard.restype = i64
            lib.orc_conv_silu.argtypes = [vp, i64, i64, i64, vp, vp, i64, vp, i64, vp, i64, vp]
            lib.orc_conv_silu.restype = None
            lib.orc_gdn_forward.argtypes = [vp, vp, vp, vp, vp, vp, vp, i64, i64, i64, i64, i64,
                                            dbl, i32, vp, vp]
            lib.orc_gdn_forward.restype = None
            lib.orc_gdn_summary.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64, i64, i32,
                                            vp, vp]
            lib.orc_gdn_summary.restype = None
            lib.orc_state_combine.argtypes = [vp, vp, vp, i64, i64, i64, i64, vp]
            lib.orc_state_combine.restype = None
            lib.orc_gates.argtypes = [vp, vp, vp, vp, i64, i64, vp, vp]
            lib.orc_gates.restype = None
            lib.orc_gated_rmsnorm.argtypes = [vp, vp, vp, dbl, i64, i64, vp]
            lib.orc_gated_rmsnorm.restype = None
            lib.orc_gdn_backward.argtypes = [vp, vp, vp, vp, vp, vp, vp, i64, i64, i64, i64, i64,
                                             dbl, i32, vp, vp, vp, vp, vp, vp, vp, vp]
            lib.orc_gdn_backward.restype = None
            lib.orc_max_threads.argtypes = []
            lib.orc_max_threads.restype = i32
            _lib = lib
    return _lib


def _f64(a):
    return None if a is None else np.ascontiguousarray(a, dtype=np.float64)


def _ptr(a):
    return None if a is None else a.ctypes.data


def max_threads() -> int:
    return int(_load().orc_max_threads())


PLAN_FIELDS = ("start_seq_idx", "end_seq_idx", "pre_num_ranks", "post_num_ranks",
               "is_first_rank", "is_last_rank", "pre_num_conv_tokens", "part_len")


def plan(cu_seqlens, n_shards: int):
    """Per-shard plan records: a list of dicts with ``local_cu`` (int64 array),
    ``local_seq`` (global sequence of each local segment) and the fields of
    PLAN_FIELDS.  Requires total % n_shards == 0."""
    cu = np.ascontiguousarray(cu_seqlens, dtype=np.int64)
    n = len(cu) - 1
    out = []
    for r in range(n_shards):
        loc = np.zeros(n + 1, dtype=np.int64)
        fields = np.zeros(8, dtype=np.int64)
        seq = np.zeros(n + 1, dtype=np.int64)
        m = _load().orc_plan_shard(cu.ctypes.data, n, n_shards, r, loc.ctypes.data,
                                   fields.ctypes.data, seq.ctypes.data)
        rec = {"local_cu": loc[:m].copy(), "local_seq": seq[:max(m - 1, 0)].copy()}
        rec.update({f: int(fields[i]) for i, f in enumerate(PLAN_FIELDS)})
        out.append(rec)
    return out


def conv_silu(x, w, bias, cu_seqlens, halo=None, halo_len: int = 0):
    """Causal depthwise conv1d + SiLU, zero history before each sequence start;
    the first sequence may continue from ``halo`` ([Kc-1, C], last row = the
    token just before, only the last ``halo_len`` rows present)."""
    x = _f64(x)
    T, C = x.shape
    w = _f64(w)
    Kc = w.shape[1]
    bias = _f64(bias)
    halo = _f64(halo)
    cu = np.ascontiguousarray(cu_seqlens, dtype=np.int64)
    y = np.empty((T, C), dtype=np.float64)
    _load().orc_conv_silu(x.ctypes.data, C, T, C, w.ctypes.data, _ptr(bias), Kc,
                          cu.ctypes.data, len(cu) - 1, _ptr(halo), int(halo_len), y.ctypes.data)
    return y


def gdn_forward(q, k, v, g, beta, h0, cu_seqlens, scale, l2norm=False, want_o=True):
    """Token recurrence.  q, k [T, Hk, K]; v [T, Hv, V]; g, beta [T, Hv];
    h0 [N, Hv, K, V] or None.  Returns (o [T, Hv, V] or None, h_final)."""
    q, k, v, g, beta, h0 = map(_f64, (q, k, v, g, beta, h0))
    T, Hk, K = k.shape
    Hv, V = v.shape[1], v.shape[2]
    cu = np.ascontiguousarray(cu_seqlens, dtype=np.int64)
    n = len(cu) - 1
    o = np.zeros((T, Hv, V), dtype=np.float64) if want_o else None
    hf = np.empty((n, Hv, K, V), dtype=np.float64)
    _load().orc_gdn_forward(q.ctypes.data, k.ctypes.data, v.ctypes.data, g.ctypes.data,
                            beta.ctypes.data, _ptr(h0), cu.ctypes.data, n, Hk, Hv, K, V,
                            float(scale), int(bool(l2norm)), _ptr(o), hf.ctypes.data)
    return o, hf


def gdn_backward(q, k, v, g, beta, h0, cu_seqlens, scale, dout, dh_final=None, l2norm=False):
    """Gradients of the token recurrence (gdn_forward) for the loss gradients
    dout [T, Hv, V] and dh_final [N, Hv, K, V] (or None): a dict with dq, dk
    [T, Hk, K] (summed over the value heads of each q/k head), dv [T, Hv, V],
    dg, dbeta [T, Hv] and dh0 [N, Hv, K, V]."""
    q, k, v, g, beta, h0, dout, dh_final = map(_f64, (q, k, v, g, beta, h0, dout, dh_final))
    T, Hk, K = k.shape
    Hv, V = v.shape[1], v.shape[2]
    cu = np.ascontiguousarray(cu_seqlens, dtype=np.int64)
    n = len(cu) - 1
    out = dict(dq=np.empty((T, Hk, K)), dk=np.empty((T, Hk, K)), dv=np.empty((T, Hv, V)),
               dg=np.empty((T, Hv)), dbeta=np.empty((T, Hv)), dh0=np.empty((n, Hv, K, V)))
    _load().orc_gdn_backward(q.ctypes.data, k.ctypes.data, v.ctypes.data, g.ctypes.data,
                             beta.ctypes.data, _ptr(h0), cu.ctypes.data, n, Hk, Hv, K, V,
                             float(scale), int(bool(l2norm)), dout.ctypes.data, _ptr(dh_final),
                             *(out[x].ctypes.data for x in ("dq", "dk", "dv", "dg", "dbeta", "dh0")))
    return out


def gdn_summary(k, v, g, beta, cu_seqlens, l2norm=False):
    """Affine summary per segment and v-head: M [N, Hv, K, K], N [N, Hv, K, V]."""
    k, v, g, beta = map(_f64, (k, v, g, beta))
    T, Hk, K = k.shape
    Hv, V = v.shape[1], v.shape[2]
    cu = np.ascontiguousarray(cu_seqlens, dtype=np.int64)
    n = len(cu) - 1
    M = np.empty((n, Hv, K, K), dtype=np.float64)
    N = np.empty((n, Hv, K, V), dtype=np.float64)
    _load().orc_gdn_summary(k.ctypes.data, v.ctypes.data, g.ctypes.data, beta.ctypes.data,
                            cu.ctypes.data, n, Hk, Hv, K, V, int(bool(l2norm)), M.ctypes.data,
                            N.ctypes.data)
    return M, N


def state_combine(M, N, S0=None):
    """state(0) = S0 or 0; state(r) = M[r-1] state(r-1) + N[r-1]; returns [P, Hv, K, V]."""
    M, N, S0 = _f64(M), _f64(N), _f64(S0)
    P, Hv, K, V = N.shape
    S_in = np.empty((P, Hv, K, V), dtype=np.float64)
    _load().orc_state_combine(M.ctypes.data, N.ctypes.data, _ptr(S0), P, Hv, K, V,
                              S_in.ctypes.data)
    return S_in


def path_forward(x, conv_w, conv_b, g, beta, h0, cu_seqlens, Hk, Hv, K, V, scale):
    """The whole path, unsharded: conv + SiLU over the fused [Q | K | V]
    channels (zero history per sequence), split, q/k L2 norm, token recurrence.
    Returns (o [T, Hv, V], h_final [N, Hv, K, V])."""
    y = conv_silu(x, conv_w, conv_b, cu_seqlens)
    T = y.shape[0]
    q = y[:, :Hk * K].reshape(T, Hk, K)
    k = y[:, Hk * K:2 * Hk * K].reshape(T, Hk, K)
    v = y[:, 2 * Hk * K:].reshape(T, Hv, V)
    return gdn_forward(q, k, v, g, beta, h0, cu_seqlens, scale, l2norm=True)


def gates(a, b, A_log, dt_bias):
    """The wrappers' gates from the raw projections: g = -exp(A_log) softplus(a +
    dt_bias), beta = sigmoid(b).  a, b [T, Hv]; A_log, dt_bias [Hv]."""
    a, b, A_log, dt_bias = map(_f64, (a, b, A_log, dt_bias))
    T, Hv = a.shape
    g = np.empty((T, Hv), dtype=np.float64)
    beta = np.empty((T, Hv), dtype=np.float64)
    _load().orc_gates(a.ctypes.data, b.ctypes.data, A_log.ctypes.data, dt_bias.ctypes.data, T, Hv,
                      g.ctypes.data, beta.ctypes.data)
    return g, beta


def gated_rmsnorm(o, z, w, eps=1e-6):
    """Gated RMS norm over the last axis: w * o / sqrt(mean(o^2) + eps) * silu(z)."""
    o, z, w = _f64(o), _f64(z), _f64(w)
    shape = o.shape
    D = shape[-1]
    rows = int(np.prod(shape[:-1]))
    y = np.empty(shape, dtype=np.float64)
    _load().orc_gated_rmsnorm(o.ctypes.data, z.ctypes.data, w.ctypes.data, float(eps), rows, D,
                              y.ctypes.data)
    return y


def layer_forward(x, conv_w, conv_b, a, b, A_log, dt_bias, z, norm_w, h0, cu_seqlens, Hk, Hv, K, V,
                  scale, eps=1e-6):
    """The wrappers' forward between the projections and the output
    projection, unsharded: gates from a and b, the path (conv + SiLU, split,
    L2 norm, recurrence), then the gated RMS norm with z.  Returns
    (y [T, Hv, V], h_final [N, Hv, K, V])."""
    g, beta = gates(a, b, A_log, dt_bias)
    o, hf = path_forward(x, conv_w, conv_b, g, beta, h0, cu_seqlens, Hk, Hv, K, V, scale)
    return gated_rmsnorm(o, z, norm_w, eps), hf
