"""Seeded synthetic workloads shared by the tests, the bench and the oracle.

This module holds no step of the Gated DeltaNet method.  It defines the
workload shapes (token counts, sequence-length mixes, head counts, dtypes,
shard counts), draws every input from the counter-based generator in
``synth.c`` and rounds it to its storage dtype.  The CUDA library and the
fp64 oracle both read exactly these arrays.

bf16 tensors are carried as ``uint16`` bit patterns (numpy has no bf16).
"""
from __future__ import annotations

import ctypes
import dataclasses
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SO = os.path.join(_HERE, "_synth.so")
_SRC = os.path.join(_HERE, "synth.c")
_lock = threading.Lock()
_lib = None

# tensor ids: one independent stream per input tensor
TID_X, TID_CONV_W, TID_CONV_B, TID_Q, TID_K, TID_V, TID_BETA, TID_G, TID_H0, TID_LEN = range(1, 11)
# the layer's raw inputs around the path: gate projections a and b, A_log,
# dt_bias, the norm gate z and the norm weight
TID_A, TID_B, TID_ALOG, TID_DTB, TID_Z, TID_NORMW = range(11, 17)
KIND_NORMAL, KIND_SIGMOID, KIND_NEG_SOFTPLUS, KIND_UNIFORM = 0, 1, 2, 3
DT_F32, DT_BF16, DT_F64 = 0, 1, 2


def build_synth(force: bool = False) -> str:
    """Compile synth.c into a shared library next to it (host code only)."""
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".{os.getpid()}.tmp"
        subprocess.run(
            ["gcc", "-O2", "-ffp-contract=off", "-fopenmp", "-fPIC", "-shared",
             "-o", tmp, _SRC, "-lm"], check=True)
        os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build_synth())
            u64, i64, i32, dbl, vp = (ctypes.c_uint64, ctypes.c_int64, ctypes.c_int,
                                      ctypes.c_double, ctypes.c_void_p)
            lib.synth_fill.argtypes = [u64, u64, i64, i64, i64, i64, i64, i32, dbl, dbl, i32, vp]
            lib.synth_fill.restype = None
            lib.synth_fill_sphere.argtypes = [u64, u64, i64, i64, i64, i64, i64, i64, i32, vp]
            lib.synth_fill_sphere.restype = None
            lib.synth_draws.argtypes = [u64, u64, i64, i64, vp]
            lib.synth_draws.restype = None
            lib.synth_key.argtypes = [u64, u64]
            lib.synth_key.restype = u64
            _lib = lib
    return _lib


_NP = {DT_F32: np.float32, DT_BF16: np.uint16, DT_F64: np.float64}


def fill(seed, tid, row_len, rows, cols, kind=KIND_NORMAL, a=0.0, b=1.0, dtype=DT_F64):
    """Elements [rows.start:rows.stop, cols.start:cols.stop] of a generated tensor."""
    r0, r1 = rows
    c0, c1 = cols
    out = np.empty((r1 - r0, c1 - c0), dtype=_NP[dtype])
    _load().synth_fill(seed, tid, row_len, r0, r1 - r0, c0, c1 - c0, kind, a, b, dtype,
                       out.ctypes.data)
    return out


def fill_sphere(seed, tid, row_len, rows, cols, group, dtype=DT_F64):
    r0, r1 = rows
    c0, c1 = cols
    assert c0 % group == 0 and (c1 - c0) % group == 0
    out = np.empty((r1 - r0, c1 - c0), dtype=_NP[dtype])
    _load().synth_fill_sphere(seed, tid, row_len, r0, r1 - r0, c0, c1 - c0, group, dtype,
                              out.ctypes.data)
    return out


def draws(seed, tid, start, n):
    out = np.empty(n, dtype=np.uint64)
    _load().synth_draws(seed, tid, start, n, out.ctypes.data)
    return out


def bf16_to_f32(u16: np.ndarray) -> np.ndarray:
    return (u16.astype(np.uint32) << 16).view(np.float32)


def as_f64(arr: np.ndarray, dtype: str) -> np.ndarray:
    """Exact fp64 values of a stored array (bf16 bits or fp32)."""
    if dtype == "bf16":
        return bf16_to_f32(arr).astype(np.float64)
    return arr.astype(np.float64)


# ----------------------------------------------------------------------------
# workload definitions
# ----------------------------------------------------------------------------

@dataclasses.dataclass
class Workload:
    name: str
    T: int
    Hk: int
    Hv: int
    dk: int
    dv: int
    dtype: str            # "f32" or "bf16": storage dtype of q/k/v/x/beta/o
    n_shards: int
    seed: int
    lengths: tuple        # sequence lengths, sum == T
    conv_k: int = 4
    g_shift: float = 0.0  # g = -softplus(N(0,1) + g_shift)
    g_zero: bool = False  # g = 0 exactly (no decay)
    h0_std: float = 0.0   # 0 -> no initial state
    conv_bias: bool = False
    w_std: float = 0.5

    @property
    def Cch(self) -> int:
        return 2 * self.Hk * self.dk + self.Hv * self.dv

    @property
    def N(self) -> int:
        return len(self.lengths)

    @property
    def dt(self) -> int:
        return DT_BF16 if self.dtype == "bf16" else DT_F32

    @property
    def scale(self) -> float:
        return self.dk ** -0.5

    def cu_seqlens(self) -> np.ndarray:
        cu = np.zeros(self.N + 1, dtype=np.int32)
        cu[1:] = np.cumsum(np.asarray(self.lengths, dtype=np.int64))
        return cu

    # ---- inputs of the whole path (raw conv input) -------------------------
    def x(self, rows=None, cols=None):
        rows = rows or (0, self.T)
        cols = cols or (0, self.Cch)
        return fill(self.seed, TID_X, self.Cch, rows, cols, dtype=self.dt)

    def conv_w(self):
        return fill(self.seed, TID_CONV_W, self.conv_k, (0, self.Cch), (0, self.conv_k),
                    b=self.w_std, dtype=self.dt)

    def conv_b(self):
        if not self.conv_bias:
            return None
        return fill(self.seed, TID_CONV_B, self.Cch, (0, 1), (0, self.Cch), b=0.5,
                    dtype=self.dt)[0]

    # ---- inputs of the chunk step (already normalised q/k) ----------------
    def q(self, rows=None, heads=None):
        return self._sphere(TID_Q, rows, heads)

    def k(self, rows=None, heads=None):
        return self._sphere(TID_K, rows, heads)

    def _sphere(self, tid, rows, heads):
        rows = rows or (0, self.T)
        h0, h1 = heads or (0, self.Hk)
        return fill_sphere(self.seed, tid, self.Hk * self.dk, rows,
                           (h0 * self.dk, h1 * self.dk), self.dk, dtype=self.dt)

    def v(self, rows=None, cols=None):
        rows = rows or (0, self.T)
        cols = cols or (0, self.Hv * self.dv)
        return fill(self.seed, TID_V, self.Hv * self.dv, rows, cols, dtype=self.dt)

    def beta(self, rows=None, heads=None):
        rows = rows or (0, self.T)
        heads = heads or (0, self.Hv)
        return fill(self.seed, TID_BETA, self.Hv, rows, heads, kind=KIND_SIGMOID, dtype=self.dt)

    def g(self, rows=None, heads=None):
        rows = rows or (0, self.T)
        heads = heads or (0, self.Hv)
        if self.g_zero:
            return np.zeros((rows[1] - rows[0], heads[1] - heads[0]), dtype=np.float32)
        return fill(self.seed, TID_G, self.Hv, rows, heads, kind=KIND_NEG_SOFTPLUS,
                    a=self.g_shift, dtype=DT_F32)

    def h0(self):
        if self.h0_std == 0.0:
            return None
        return fill(self.seed, TID_H0, self.Hv * self.dk * self.dv, (0, self.N),
                    (0, self.Hv * self.dk * self.dv), b=self.h0_std,
                    dtype=DT_F32).reshape(self.N, self.Hv, self.dk, self.dv)

    # ---- the layer's raw inputs (gates from projections, gated norm) -----
    # a, b ~ N(0, 1) per (token, v-head) (so beta = sigmoid(b) has the
    # recipe's distribution); A_log = log U[1, 16] and dt_bias ~ N(0, 1) per
    # v-head; z ~ N(0, 1) [T, Hv, dv]; norm weight ~ 1 + N(0, 0.1^2) [dv]
    def a_proj(self, rows=None):
        rows = rows or (0, self.T)
        return fill(self.seed, TID_A, self.Hv, rows, (0, self.Hv), dtype=self.dt)

    def b_proj(self, rows=None):
        rows = rows or (0, self.T)
        return fill(self.seed, TID_B, self.Hv, rows, (0, self.Hv), dtype=self.dt)

    def A_log(self):
        u = fill(self.seed, TID_ALOG, self.Hv, (0, 1), (0, self.Hv), kind=KIND_UNIFORM, a=1.0,
                 b=15.0)[0]
        return np.log(u).astype(np.float32)

    def dt_bias(self):
        return fill(self.seed, TID_DTB, self.Hv, (0, 1), (0, self.Hv), dtype=DT_F32)[0]

    def z(self, rows=None):
        rows = rows or (0, self.T)
        return fill(self.seed, TID_Z, self.Hv * self.dv, rows, (0, self.Hv * self.dv), dtype=self.dt)

    def norm_w(self):
        return fill(self.seed, TID_NORMW, self.dv, (0, 1), (0, self.dv), a=1.0, b=0.1, dtype=self.dt)[0]

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


def lengths_uniform(seed, T, lo, hi):
    """Lengths ~ U{lo..hi} drawn until they cover T; the last one is truncated."""
    out, total, i = [], 0, 0
    while total < T:
        u = fill(seed, TID_LEN, 1, (i, i + 1), (0, 1), kind=KIND_UNIFORM)[0, 0]
        n = lo + int(np.floor(u * (hi - lo + 1)))
        n = min(n, T - total)
        out.append(n)
        total += n
        i += 1
    return tuple(out)


def lengths_geometric(seed, T, p, lo, hi):
    """Lengths ~ Geometric(p) on {1,2,...} (inverse CDF), clipped to [lo, hi]."""
    out, total, i = [], 0, 0
    lq = np.log1p(-p)
    while total < T:
        u = fill(seed, TID_LEN, 1, (i, i + 1), (0, 1), kind=KIND_UNIFORM)[0, 0]
        n = int(np.ceil(np.log(u) / lq))
        n = max(lo, min(hi, n))
        n = min(n, T - total)
        out.append(n)
        total += n
        i += 1
    return tuple(out)


def tiny(**kw) -> Workload:
    """1 sequence of 256 tokens, 2 heads, d=32, fp32, 2 virtual shards, seed 0."""
    return Workload("tiny", 256, 2, 2, 32, 32, "f32", kw.pop("n_shards", 2), kw.pop("seed", 0),
                    (256,), **kw)


def packed_varlen(T: int = 32768, **kw) -> Workload:
    """Packed varlen: lengths ~ U{512..8192}; 16 qk heads, 32 v heads, d=128, bf16, P=1."""
    seed = kw.pop("seed", 1)
    return Workload("packed_varlen", T, 16, 32, 128, 128, "bf16", kw.pop("n_shards", 1), seed,
                    lengths_uniform(seed, T, 512, 8192), **kw)


def long_seq(T: int = 131072, **kw) -> Workload:
    """One long sequence, 16 heads, d=128, bf16, 8 virtual shards."""
    return Workload("long", T, 16, 16, 128, 128, "bf16", kw.pop("n_shards", 8),
                    kw.pop("seed", 2), (T,), **kw)


def ragged(T: int = 65536, **kw) -> Workload:
    """Geometric(mean 300) lengths in [1, 4096], 16 heads, d=128, bf16, 16 shards."""
    seed = kw.pop("seed", 3)
    return Workload("ragged", T, 16, 16, 128, 128, "bf16", kw.pop("n_shards", 16), seed,
                    lengths_geometric(seed, T, 1.0 / 300.0, 1, 4096), **kw)


def million(T: int = 1048576, **kw) -> Workload:
    """One 1M-token sequence, 32 heads, d=128, bf16, 64 shards, h0 ~ N(0, 0.02^2),
    g = -softplus(N(0,1) + 2)."""
    return Workload("million", T, 32, 32, 128, 128, "bf16", kw.pop("n_shards", 64),
                    kw.pop("seed", 4), (T,), g_shift=kw.pop("g_shift", 2.0),
                    h0_std=kw.pop("h0_std", 0.02), **kw)


CONFIGS = {"tiny": tiny, "packed_varlen": packed_varlen, "long": long_seq,
           "ragged": ragged, "million": million}
