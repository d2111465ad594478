"""Thin ctypes binding of libgdncp (include/gdn_cp.h).

Argument marshalling only: every step of the computation runs in the CUDA
kernels of libgdncp.  PyTorch provides device memory and the current CUDA
stream.  There is no CPU fallback: if the library is missing or a call
fails, an exception is raised.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libgdncp.so")

GDN_F32, GDN_BF16 = 0, 1
GDN_QK_L2NORM = 1
PLAN_FIELDS = ("local_num_seqs", "start_seq_idx", "end_seq_idx", "pre_num_ranks",
               "post_num_ranks", "is_first_rank", "is_last_rank", "pre_num_conv_tokens",
               "seg_offset")
STATUS = {0: "GDN_OK", 1: "GDN_ERR_INVALID_ARG", 2: "GDN_ERR_UNSUPPORTED_SHAPE",
          3: "GDN_ERR_DTYPE", 4: "GDN_ERR_NOT_DIVISIBLE", 5: "GDN_ERR_SHARD_TOO_SHORT",
          6: "GDN_ERR_BAD_CU_SEQLENS", 7: "GDN_ERR_TIMEOUT", 8: "GDN_ERR_CUDA",
          9: "GDN_ERR_WORKSPACE"}

# exported symbols and their ctypes signatures
_vp, _i32, _i64, _u32, _f32, _sz = (ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64,
                                    ctypes.c_uint32, ctypes.c_float, ctypes.c_size_t)
SIGNATURES = {
    "gdn_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "gdn_last_error": (ctypes.c_char_p, []),
    "gdn_device_timeouts": (ctypes.c_int, [_vp, ctypes.c_int]),
    "gdn_debug_set_handover": (ctypes.c_int, [_i64, ctypes.c_int]),
    "gdn_debug_set_split": (ctypes.c_int, [_i32]),
    "gdn_debug_set_phase_events": (ctypes.c_int, [_vp, _i32]),
    "gdn_cp_plan_words": (_i64, [_i32, _i32]),
    "gdn_cp_plan": (ctypes.c_int, [_vp, _i32, _i32, _vp, _vp]),
    "gdn_conv_silu": (ctypes.c_int, [_vp, _i64, ctypes.c_int, _i32, _i32, _vp, _vp, _i32, _vp,
                                     _i32, _vp, _i32, _vp, _i64, _vp]),
    "gdn_chunk_fwd": (ctypes.c_int, [_vp, _vp, _vp, _i64, _i64, _i64, ctypes.c_int, _vp, _vp,
                                     _vp, _vp, _i32, _i32, _i32, _i32, _i32, _i32, _f32, _u32,
                                     _vp, _vp, _vp, ctypes.c_size_t, _vp]),
    "gdn_chunk_fwd_heads": (ctypes.c_int, [_vp, _vp, _vp, ctypes.c_int, _vp, _vp, _vp, _vp, _i32, _i32, _i32,
                                           _i32, _i32, _i32, _f32, _u32, _vp, _vp, _vp, ctypes.c_size_t, _vp]),
    "gdn_to_head_major": (ctypes.c_int, [_vp, _i64, ctypes.c_int, _i32, _i32, _i32, _vp, _vp]),
    "gdn_to_token_major": (ctypes.c_int, [_vp, ctypes.c_int, _i32, _i32, _i32, _vp, _i64, _vp]),
    "gdn_chunk_fwd_workspace_size": (ctypes.c_size_t, [_i32, _i32, _i32, _i32, ctypes.c_int]),
    "gdn_chunk_bwd_workspace_size": (ctypes.c_size_t, [_i32, _i32, _i32, _i32, _i32, _i32]),
    "gdn_shard_bwd_workspace_size": (ctypes.c_size_t, [_i32, _i32, _i32, _i32, _i32, _i32, _i32]),
    "gdn_shard_bwd": (ctypes.c_int, [_vp, _vp, _vp, _i64, _i64, _i64, ctypes.c_int, _vp, _vp, _vp, _vp, _vp,
                                     _vp, _i32, _i32, _i32, _i32, _i32, _i32, _f32, _u32, _i32, _vp, _vp, _vp,
                                     _vp, _vp, _vp, _vp, ctypes.c_size_t, _vp, _vp]),
    "gdn_chunk_bwd": (ctypes.c_int, [_vp, _vp, _vp, _i64, _i64, _i64, ctypes.c_int, _vp, _vp, _vp, _vp, _vp,
                                     _vp, _i32, _i32, _i32, _i32, _i32, _i32, _f32, _u32, _vp, _vp, _vp, _vp,
                                     _vp, _vp, _vp, ctypes.c_size_t, _vp]),
    "gdn_chunk_summary": (ctypes.c_int, [_vp, _vp, _i64, _i64, ctypes.c_int, _vp, _vp, _vp,
                                         _i32, _i32, _i32, _i32, _i32, _i32, _u32, _vp, _vp,
                                         _vp]),
    "gdn_state_combine": (ctypes.c_int, [_vp, _vp, _vp, _i32, _i32, _i32, _i32, _vp, _vp]),
    "gdn_shard_fwd_workspace_size": (_sz, [_i32, _i32, _i32, _i32, _i32, _i32, _i32,
                                           ctypes.c_int]),
    "gdn_shard_fwd_workspace_min_size": (_sz, [_i32, _i32, _i32, _i32, _i32, _i32, _i32,
                                               ctypes.c_int]),
    "gdn_shard_fwd": (ctypes.c_int, [_vp, _vp, _vp, _i32, _vp, _vp, _vp, _vp, _i32, _i32, _i32,
                                     _i32, _i32, _i32, _f32, _u32, _i32, ctypes.c_int, _vp, _sz,
                                     _vp, _vp, _vp, _vp]),
    "gdn_layer_fwd": (ctypes.c_int, [_vp, _vp, _vp, _i32, _vp, _vp, _vp, _vp, _vp, _i64, _vp, _f32, _vp, _vp,
                                     _i32, _i32, _i32, _i32, _i32, _i32, _f32, _u32, _i32, ctypes.c_int, _vp, _sz,
                                     _vp, _vp, _vp, _vp]),
    "gdn_shard_fwd_noalloc": (ctypes.c_int, [_vp, _vp, _vp, _i32, _vp, _vp, _vp, _vp, _i32, _i32,
                                             _i32, _i32, _i32, _i32, _f32, _u32, _i32,
                                             ctypes.c_int, _vp, _vp, _vp, _vp]),
}
NOALLOC_SCRATCH_BYTES = 32 << 20

_lock = threading.Lock()
_lib = None


class GdnError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{STATUS.get(status, status)}: {msg}")
        self.status = status


def load():
    """Load libgdncp.so (built by build.build_library()); raise if missing."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"{LIB_PATH} is missing: build it first "
                                   "(linear_attention_sequence_device_gb300.build.build_library)")
            lib = ctypes.CDLL(LIB_PATH)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib


def _check(st: int):
    if st != 0:
        raise GdnError(st, load().gdn_last_error().decode())


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _dt(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return GDN_BF16
    if t.dtype == torch.float32:
        return GDN_F32
    raise TypeError(f"unsupported dtype {t.dtype}")


def _need(t, name, dtype=None):
    if t is None:
        return
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")


def _row_stride(t: torch.Tensor, name: str) -> int:
    """Token stride of a [T, H, d] view whose (H, d) part is dense."""
    if t.dim() != 3 or t.stride(2) != 1 or t.stride(1) != t.shape[2]:
        raise ValueError(f"{name} must be a [T, H, d] view with dense heads")
    return t.stride(0)


# ----------------------------------------------------------------------------
# entry points
# ----------------------------------------------------------------------------

def device_timeouts(reset: bool = False) -> int:
    """Bounded device waits that expired since load / the last reset (syncs)."""
    n = ctypes.c_int32(0)
    _check(load().gdn_device_timeouts(ctypes.byref(n), 1 if reset else 0))
    return n.value


def debug_set_handover(wait_ns: int = 1_000_000_000, publish: bool = True):
    """Testing hook: bound of the split-item hand-over wait and whether first
    halves publish their final state (see gdn_cp.h); the defaults restore
    normal operation."""
    _check(load().gdn_debug_set_handover(int(wait_ns), 1 if publish else 0))


def debug_set_split(enable: bool = True):
    """Testing hook: work-queue splitting of items on or off (see gdn_cp.h);
    the default restores normal operation."""
    _check(load().gdn_debug_set_split(1 if enable else 0))


def debug_set_phase_events(events=None):
    """Profiling hook: torch.cuda.Event objects (already recorded once, so
    that their handles exist) that gdn_shard_fwd records between its phases
    on this thread; None turns it off."""
    events = list(events or [])
    arr = (ctypes.c_void_p * max(1, len(events)))(*[ctypes.c_void_p(e.cuda_event) for e in events])
    _check(load().gdn_debug_set_phase_events(arr, len(events)))


def plan_words(num_seqs: int, n_shards: int) -> int:
    return int(load().gdn_cp_plan_words(num_seqs, n_shards))


def gdn_cp_plan(cu_seqlens: torch.Tensor, n_shards: int, out: torch.Tensor | None = None):
    """Device shard plan; returns the int32 plan words (see gdn_cp.h)."""
    _need(cu_seqlens, "cu_seqlens", torch.int32)
    n = cu_seqlens.numel() - 1
    if out is None:
        out = torch.empty(plan_words(n, n_shards), dtype=torch.int32, device=cu_seqlens.device)
    _check(load().gdn_cp_plan(_p(cu_seqlens), n, n_shards, _p(out), _stream()))
    return out


def decode_plan(plan, num_seqs: int, n_shards: int):
    """Host view of plan words: (status, [per-shard dict with local_cu and
    local_seq, the global sequence of each local segment])."""
    w = plan.cpu().tolist() if isinstance(plan, torch.Tensor) else list(plan)
    recs = []
    base_cu = 1 + n_shards * len(PLAN_FIELDS)
    for r in range(n_shards):
        rec = dict(zip(PLAN_FIELDS, w[1 + r * len(PLAN_FIELDS):1 + (r + 1) * len(PLAN_FIELDS)]))
        off = base_cu + r * (num_seqs + 1)
        rec["local_cu"] = w[off:off + rec["local_num_seqs"] + 1]
        soff = base_cu + (n_shards + r) * (num_seqs + 1)
        rec["local_seq"] = w[soff:soff + rec["local_num_seqs"]]
        recs.append(rec)
    return w[0], recs


def gdn_conv_silu(x, w, bias, cu_seqlens, halo=None, halo_len: int = 0, out=None):
    """Causal depthwise conv1d + SiLU; x [T, C] (row-strided view allowed)."""
    for t, n in ((x, "x"), (w, "w"), (bias, "bias"), (halo, "halo")):
        _need(t, n, x.dtype)
    _need(cu_seqlens, "cu_seqlens", torch.int32)
    T, C = x.shape
    if x.stride(1) != 1:
        raise ValueError("x must have unit channel stride")
    w = w.contiguous()
    if out is None:
        out = torch.empty((T, C), dtype=x.dtype, device=x.device)
    _check(load().gdn_conv_silu(_p(x), x.stride(0), _dt(x), T, C, _p(w), _p(bias), w.shape[1],
                                _p(cu_seqlens), cu_seqlens.numel() - 1,
                                _p(None if halo is None else halo.contiguous()), halo_len,
                                _p(out), out.stride(0), _stream()))
    return out


def gdn_chunk_fwd(q, k, v, g, beta, cu_seqlens, h0=None, scale=None, l2norm=False,
                  output_final_state=True, out=None, workspace=None):
    """q, k [T, Hk, dk]; v [T, Hv, dv] (token-strided views allowed); g [T, Hv]
    fp32; beta [T, Hv]; h0 [N, Hv, dk, dv] fp32.  Returns (o, h_final).
    workspace: a uint8 device tensor of at least chunk_fwd_workspace_size
    bytes, reused across calls; allocated per call when None; False for none
    (longest-first job order only)."""
    dt = q.dtype
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (beta, "beta")):
        _need(t, n, dt)
    _need(g, "g", torch.float32)
    _need(h0, "h0", torch.float32)
    _need(cu_seqlens, "cu_seqlens", torch.int32)
    T, Hk, dk = q.shape
    Hv, dv = v.shape[1], v.shape[2]
    N = cu_seqlens.numel() - 1
    scale = dk ** -0.5 if scale is None else scale
    o = torch.empty((T, Hv, dv), dtype=dt, device=q.device) if out is None else out
    hf = torch.empty((N, Hv, dk, dv), dtype=torch.float32, device=q.device) \
        if output_final_state else None
    lib = load()
    if workspace is None:
        ws = torch.empty(max(lib.gdn_chunk_fwd_workspace_size(N, Hv, dk, dv, _dt(q)), 16), dtype=torch.uint8,
                         device=q.device)
    else:
        ws = workspace if workspace is not False else None
    _check(lib.gdn_chunk_fwd(_p(q), _p(k), _p(v), _row_stride(q, "q"), _row_stride(k, "k"),
                             _row_stride(v, "v"), _dt(q), _p(g.contiguous()),
                             _p(beta.contiguous()), _p(None if h0 is None else h0.contiguous()),
                             _p(cu_seqlens), N, T, Hk, Hv, dk, dv, float(scale),
                             GDN_QK_L2NORM if l2norm else 0, _p(o), _p(hf), _p(ws),
                             0 if ws is None else ws.numel(), _stream()))
    return o, hf


def gdn_chunk_bwd(q, k, v, g, beta, cu_seqlens, dout, h0=None, dh_final=None, scale=None, l2norm=False,
                  workspace=None, n_shards=None, want_plan=False):
    """Gradients of gdn_chunk_fwd's outputs (o, h_final) w.r.t. its inputs, for
    the loss gradients dout [T, Hv, dv] (dtype of v) and dh_final [N, Hv, dk,
    dv] fp32 (None: zero).  Returns a dict of fp32 tensors dq, dk [T, Hk, dk],
    dv [T, Hv, dv], dg, dbeta [T, Hv] and dh0 [N, Hv, dk, dv].  workspace: a
    uint8 device tensor of at least chunk_bwd_workspace_size bytes (allocated
    per call when None).  n_shards: run it on that many virtual shards
    (gdn_shard_bwd; want_plan also returns the plan words as "plan")."""
    dt = q.dtype
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (beta, "beta"), (dout, "dout")):
        _need(t, n, dt)
    _need(g, "g", torch.float32)
    _need(h0, "h0", torch.float32)
    _need(dh_final, "dh_final", torch.float32)
    _need(cu_seqlens, "cu_seqlens", torch.int32)
    T, Hk, dk = q.shape
    Hv, dv = v.shape[1], v.shape[2]
    N = cu_seqlens.numel() - 1
    scale = dk ** -0.5 if scale is None else scale
    dev = q.device
    f32 = torch.float32
    out = dict(dq=torch.empty((T, Hk, dk), dtype=f32, device=dev), dk=torch.empty((T, Hk, dk), dtype=f32, device=dev),
               dv=torch.empty((T, Hv, dv), dtype=f32, device=dev), dg=torch.empty((T, Hv), dtype=f32, device=dev),
               dbeta=torch.empty((T, Hv), dtype=f32, device=dev),
               dh0=torch.empty((N, Hv, dk, dv), dtype=f32, device=dev))
    lib = load()
    if n_shards is not None:
        if workspace is None:
            workspace = torch.empty(max(lib.gdn_shard_bwd_workspace_size(T, N, n_shards, Hk, Hv, dk, dv), 256),
                                    dtype=torch.uint8, device=dev)
        plan = torch.empty(plan_words(N, n_shards), dtype=torch.int32, device=dev) if want_plan else None
        _check(lib.gdn_shard_bwd(_p(q), _p(k), _p(v), _row_stride(q, "q"), _row_stride(k, "k"), _row_stride(v, "v"),
                                 _dt(q), _p(g.contiguous()), _p(beta.contiguous()),
                                 _p(None if h0 is None else h0.contiguous()), _p(dout.contiguous()),
                                 _p(None if dh_final is None else dh_final.contiguous()), _p(cu_seqlens), N, T, Hk,
                                 Hv, dk, dv, float(scale), GDN_QK_L2NORM if l2norm else 0, int(n_shards),
                                 *(_p(out[x]) for x in ("dq", "dk", "dv", "dg", "dbeta", "dh0")),
                                 _p(workspace), workspace.numel(), _p(plan), _stream()))
        if want_plan:
            out["plan"] = plan
        return out
    if workspace is None:
        workspace = torch.empty(max(lib.gdn_chunk_bwd_workspace_size(T, N, Hk, Hv, dk, dv), 256), dtype=torch.uint8,
                                device=dev)
    _check(lib.gdn_chunk_bwd(_p(q), _p(k), _p(v), _row_stride(q, "q"), _row_stride(k, "k"), _row_stride(v, "v"),
                             _dt(q), _p(g.contiguous()), _p(beta.contiguous()),
                             _p(None if h0 is None else h0.contiguous()), _p(dout.contiguous()),
                             _p(None if dh_final is None else dh_final.contiguous()), _p(cu_seqlens), N, T, Hk, Hv,
                             dk, dv, float(scale), GDN_QK_L2NORM if l2norm else 0,
                             *(_p(out[x]) for x in ("dq", "dk", "dv", "dg", "dbeta", "dh0")),
                             _p(workspace), workspace.numel(), _stream()))
    return out


def chunk_bwd_workspace_size(T, num_seqs, Hk, Hv, dk, dv) -> int:
    return int(load().gdn_chunk_bwd_workspace_size(T, num_seqs, Hk, Hv, dk, dv))


def to_head_major(x, out=None):
    """[T, H, d] (token-strided view with dense heads) -> dense [H, T, d]."""
    _need(x, "x")
    T, H, d = x.shape
    ld = _row_stride(x, "x")
    y = torch.empty((H, T, d), dtype=x.dtype, device=x.device) if out is None else out
    _check(load().gdn_to_head_major(_p(x), ld, _dt(x), T, H, d, _p(y), _stream()))
    return y


def to_token_major(y, out=None):
    """Dense [H, T, d] -> [T, H, d] (out may be a token-strided view)."""
    _need(y, "y")
    H, T, d = y.shape
    x = torch.empty((T, H, d), dtype=y.dtype, device=y.device) if out is None else out
    _check(load().gdn_to_token_major(_p(y.contiguous()), _dt(y), T, H, d, _p(x), _row_stride(x, "out"),
                                     _stream()))
    return x


def gdn_chunk_fwd_heads(q, k, v, g, beta, cu_seqlens, h0=None, scale=None, l2norm=False, out=None,
                        workspace=None):
    """Head-major chunked forward: q, k [Hk, T, dk], v [Hv, T, dv] dense;
    g, beta [T, Hv].  Returns (o [Hv, T, dv], h_final [N, Hv, dk, dv])."""
    dt = q.dtype
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (beta, "beta")):
        _need(t, n, dt)
    _need(g, "g", torch.float32)
    _need(h0, "h0", torch.float32)
    _need(cu_seqlens, "cu_seqlens", torch.int32)
    Hk, T, dk = q.shape
    Hv, dv = v.shape[0], v.shape[2]
    N = cu_seqlens.numel() - 1
    scale = dk ** -0.5 if scale is None else scale
    o = torch.empty((Hv, T, dv), dtype=dt, device=q.device) if out is None else out
    hf = torch.empty((N, Hv, dk, dv), dtype=torch.float32, device=q.device)
    lib = load()
    if workspace is None:
        ws = torch.empty(max(lib.gdn_chunk_fwd_workspace_size(N, Hv, dk, dv, _dt(q)), 16), dtype=torch.uint8,
                         device=q.device)
    else:
        ws = workspace if workspace is not False else None
    _check(lib.gdn_chunk_fwd_heads(_p(q.contiguous()), _p(k.contiguous()), _p(v.contiguous()), _dt(q),
                                   _p(g.contiguous()), _p(beta.contiguous()),
                                   _p(None if h0 is None else h0.contiguous()), _p(cu_seqlens), N, T, Hk, Hv, dk,
                                   dv, float(scale), GDN_QK_L2NORM if l2norm else 0, _p(o), _p(hf), _p(ws),
                                   0 if ws is None else ws.numel(), _stream()))
    return o, hf


def chunk_fwd_workspace_size(N, Hv, dk, dv, dtype):
    """Bytes of the optional gdn_chunk_fwd workspace."""
    code = {torch.bfloat16: GDN_BF16, torch.float32: GDN_F32}[dtype]
    return load().gdn_chunk_fwd_workspace_size(N, Hv, dk, dv, code)


def gdn_chunk_summary(k, v, g, beta, cu_seqlens, l2norm=False):
    """Per sequence: (M [N, Hv, dk, dk], N [N, Hv, dk, dv]) with S_end = M S_start + N."""
    dt = k.dtype
    for t, n in ((k, "k"), (v, "v"), (beta, "beta")):
        _need(t, n, dt)
    _need(g, "g", torch.float32)
    T, Hk, dk = k.shape
    Hv, dv = v.shape[1], v.shape[2]
    n = cu_seqlens.numel() - 1
    M = torch.empty((n, Hv, dk, dk), dtype=torch.float32, device=k.device)
    Nn = torch.empty((n, Hv, dk, dv), dtype=torch.float32, device=k.device)
    _check(load().gdn_chunk_summary(_p(k), _p(v), _row_stride(k, "k"), _row_stride(v, "v"),
                                    _dt(k), _p(g.contiguous()), _p(beta.contiguous()),
                                    _p(cu_seqlens), n, T, Hk, Hv, dk, dv,
                                    GDN_QK_L2NORM if l2norm else 0, _p(M), _p(Nn), _stream()))
    return M, Nn


def gdn_state_combine(M, N, S0=None):
    """S_in[0] = S0 or 0; S_in[r] = M[r-1] S_in[r-1] + N[r-1]."""
    for t, n in ((M, "M"), (N, "N"), (S0, "S0")):
        _need(t, n, torch.float32)
    P, Hv, dk, dv = N.shape
    S_in = torch.empty_like(N)
    _check(load().gdn_state_combine(_p(M.contiguous()), _p(N.contiguous()),
                                    _p(None if S0 is None else S0.contiguous()), P, Hv, dk, dv,
                                    _p(S_in), _stream()))
    return S_in


def shard_fwd_workspace_size(T, num_seqs, n_shards, Hk, Hv, dk, dv, dtype) -> int:
    return int(load().gdn_shard_fwd_workspace_size(T, num_seqs, n_shards, Hk, Hv, dk, dv,
                                                   GDN_BF16 if dtype == torch.bfloat16 else GDN_F32))


def shard_fwd_workspace_min_size(T, num_seqs, n_shards, Hk, Hv, dk, dv, dtype) -> int:
    return int(load().gdn_shard_fwd_workspace_min_size(T, num_seqs, n_shards, Hk, Hv, dk, dv,
                                                   GDN_BF16 if dtype == torch.bfloat16 else GDN_F32))


def gdn_shard_fwd(x, conv_w, conv_b, g, beta, cu_seqlens, Hk, Hv, dk, dv, n_shards, h0=None,
                  scale=None, l2norm=True, workspace=None, out=None, h_final=True,
                  want_plan=False):
    """The whole path on n_shards virtual shards.  x [T, 2*Hk*dk + Hv*dv].
    h_final: True (allocate), False (skip) or an output tensor [N, Hv, dk, dv].
    Returns (o [T, Hv, dv], h_final [N, Hv, dk, dv] or None, plan words or None)."""
    dt = x.dtype
    for t, n in ((x, "x"), (conv_w, "conv_w"), (conv_b, "conv_b"), (beta, "beta")):
        _need(t, n, dt)
    _need(g, "g", torch.float32)
    _need(h0, "h0", torch.float32)
    _need(cu_seqlens, "cu_seqlens", torch.int32)
    T = x.shape[0]
    N = cu_seqlens.numel() - 1
    scale = dk ** -0.5 if scale is None else scale
    ws_bytes = shard_fwd_workspace_size(T, N, n_shards, Hk, Hv, dk, dv, dt)
    if workspace is None:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=x.device)
    o = torch.empty((T, Hv, dv), dtype=dt, device=x.device) if out is None else out
    if isinstance(h_final, torch.Tensor):
        _need(h_final, "h_final", torch.float32)
        hf = h_final
    else:
        hf = torch.empty((N, Hv, dk, dv), dtype=torch.float32, device=x.device) if h_final else None
    plan = torch.empty(plan_words(N, n_shards), dtype=torch.int32, device=x.device) \
        if want_plan else None
    _check(load().gdn_shard_fwd(_p(x.contiguous()), _p(conv_w.contiguous()), _p(conv_b),
                                conv_w.shape[1], _p(g.contiguous()), _p(beta.contiguous()),
                                _p(None if h0 is None else h0.contiguous()), _p(cu_seqlens), N,
                                T, Hk, Hv, dk, dv, float(scale), GDN_QK_L2NORM if l2norm else 0,
                                n_shards, _dt(x), _p(workspace), workspace.numel(), _p(o), _p(hf),
                                _p(plan), _stream()))
    return o, hf, plan


def gdn_layer_fwd(x, conv_w, conv_b, a, b, A_log, dt_bias, z, norm_w, cu_seqlens, Hk, Hv, dk, dv,
                  n_shards, h0=None, scale=None, eps=1e-6, l2norm=True, workspace=None, out=None,
                  h_final=True, want_plan=False):
    """The layer between its projections: gates from a and b, the path on
    n_shards virtual shards, the gated RMS norm with z (None: no norm).
    x [T, Cch]; a, b [T, Hv]; A_log, dt_bias [Hv] fp32; z [T, Hv, dv] (dense
    heads, token stride free); norm_w [dv].  Returns (y, h_final, plan)."""
    dt = x.dtype
    for t, n in ((x, "x"), (conv_w, "conv_w"), (conv_b, "conv_b"), (a, "a"), (b, "b"), (z, "z"),
                 (norm_w, "norm_w")):
        _need(t, n, dt)
    _need(A_log, "A_log", torch.float32)
    _need(dt_bias, "dt_bias", torch.float32)
    _need(h0, "h0", torch.float32)
    _need(cu_seqlens, "cu_seqlens", torch.int32)
    T = x.shape[0]
    N = cu_seqlens.numel() - 1
    scale = dk ** -0.5 if scale is None else scale
    if workspace is None:
        workspace = torch.empty(shard_fwd_workspace_size(T, N, n_shards, Hk, Hv, dk, dv, dt), dtype=torch.uint8,
                                device=x.device)
    y = torch.empty((T, Hv, dv), dtype=dt, device=x.device) if out is None else out
    if isinstance(h_final, torch.Tensor):
        hf = h_final
    else:
        hf = torch.empty((N, Hv, dk, dv), dtype=torch.float32, device=x.device) if h_final else None
    plan = torch.empty(plan_words(N, n_shards), dtype=torch.int32, device=x.device) if want_plan else None
    ldz = 0
    if z is not None:
        z3 = z.view(T, Hv, dv) if z.dim() == 2 else z
        ldz = _row_stride(z3, "z")
    _check(load().gdn_layer_fwd(_p(x.contiguous()), _p(conv_w.contiguous()), _p(conv_b), conv_w.shape[1],
                                _p(a.contiguous()), _p(b.contiguous()), _p(A_log.contiguous()),
                                _p(dt_bias.contiguous()), _p(z), ldz,
                                _p(None if norm_w is None else norm_w.contiguous()), float(eps),
                                _p(None if h0 is None else h0.contiguous()), _p(cu_seqlens), N, T, Hk, Hv, dk,
                                dv, float(scale), GDN_QK_L2NORM if l2norm else 0, n_shards, _dt(x),
                                _p(workspace), workspace.numel(), _p(y), _p(hf), _p(plan), _stream()))
    return y, hf, plan


def gdn_shard_fwd_noalloc(x, conv_w, conv_b, g, beta, cu_seqlens, Hk, Hv, dk, dv, n_shards,
                          h0=None, scale=None, l2norm=True, out=None, h_final=True):
    """gdn_shard_fwd for callers that cannot allocate device memory: the
    library's fixed 32 MiB scratch array replaces the workspace (see
    gdn_cp.h).  This wrapper itself only allocates the outputs when they are
    not given.  Returns (o, h_final or None)."""
    dt = x.dtype
    for t, n in ((x, "x"), (conv_w, "conv_w"), (conv_b, "conv_b"), (beta, "beta")):
        _need(t, n, dt)
    _need(g, "g", torch.float32)
    _need(h0, "h0", torch.float32)
    _need(cu_seqlens, "cu_seqlens", torch.int32)
    T = x.shape[0]
    N = cu_seqlens.numel() - 1
    scale = dk ** -0.5 if scale is None else scale
    o = torch.empty((T, Hv, dv), dtype=dt, device=x.device) if out is None else out
    if isinstance(h_final, torch.Tensor):
        hf = h_final
    else:
        hf = torch.empty((N, Hv, dk, dv), dtype=torch.float32, device=x.device) if h_final else None
    _check(load().gdn_shard_fwd_noalloc(_p(x.contiguous()), _p(conv_w.contiguous()), _p(conv_b),
                                        conv_w.shape[1], _p(g.contiguous()), _p(beta.contiguous()),
                                        _p(None if h0 is None else h0.contiguous()),
                                        _p(cu_seqlens), N, T, Hk, Hv, dk, dv, float(scale),
                                        GDN_QK_L2NORM if l2norm else 0, n_shards, _dt(x), _p(o),
                                        _p(hf), None, _stream()))
    return o, hf
