"""Independent fp64 numpy restatement of the chunked (C = 64) gated delta rule
in WY/UT form, as the hyper-parallel page ``linear_attention_context_parallel.py``
lays it out (``_prepare_gdn_chunks_for_summary``, ``_run_prepared_gdn_chunks``,
``_compute_gdn_state_summary_from_prepared``).

Used only to pin the token-by-token oracle: the two forms share no code and
agree to rounding because the chunk form is exact for the recurrence.
One sequence, one head at a time; q, k [L, K], v [L, V], g, beta [L].
"""
from __future__ import annotations

import numpy as np


def _prepare(q, k, v, g, beta, C, scale):
    L, K = k.shape
    pad = (-L) % C
    # zero padding: padded rows have beta = 0 and g = 0, so they change nothing
    q, k, v = (np.pad(a, ((0, pad), (0, 0))) for a in (q, k, v))
    g, beta = np.pad(g, (0, pad)), np.pad(beta, (0, pad))
    n = (L + pad) // C
    q = (q * scale).reshape(n, C, K)
    k = k.reshape(n, C, K)
    v = v.reshape(n, C, -1)
    beta = beta.reshape(n, C)
    G = np.cumsum(g.reshape(n, C), axis=1)                     # in-chunk gate prefix
    diff = G[:, :, None] - G[:, None, :]
    lower_incl = np.tril(np.ones((C, C), dtype=bool))
    gamma = np.where(lower_incl, np.exp(np.where(lower_incl, diff, 0.0)), 0.0)
    kb = k * beta[:, :, None]
    vb = v * beta[:, :, None]
    # strictly-lower part of -(beta_i k_i.k_j Gamma_ij), then forward substitution
    A = -(kb @ k.transpose(0, 2, 1)) * gamma
    A = np.where(np.tril(np.ones((C, C), dtype=bool), -1), A, 0.0)
    for i in range(1, C):
        A[:, i, :i] = A[:, i, :i] + np.einsum("nm,nmj->nj", A[:, i, :i], A[:, :i, :i])
    Tm = A + np.eye(C)                                          # (I + L)^-1
    U = Tm @ vb
    W = Tm @ (kb * np.exp(G)[:, :, None])
    return q, k, U, W, G, gamma, n


def chunk_forward(q, k, v, g, beta, h0=None, C=64, scale=None):
    """Returns (o [L, V], final state [K, V])."""
    L, K = k.shape
    V = v.shape[1]
    scale = K ** -0.5 if scale is None else scale
    qc, kc, U, W, G, gamma, n = _prepare(q, k, v, g, beta, C, scale)
    S = np.zeros((K, V)) if h0 is None else np.array(h0, dtype=np.float64)
    o = np.zeros((n, C, V))
    for c in range(n):
        v_new = U[c] - W[c] @ S
        o[c] = (qc[c] * np.exp(G[c])[:, None]) @ S + ((qc[c] @ kc[c].T) * gamma[c]) @ v_new
        decay_k = kc[c] * np.exp(G[c, -1] - G[c])[:, None]
        S = np.exp(G[c, -1]) * S + decay_k.T @ v_new
    return o.reshape(n * C, V)[:L], S


def chunk_summary(k, v, g, beta, C=64):
    """(M [K, K], N [K, V]) with state_out = M state_in + N."""
    L, K = k.shape
    V = v.shape[1]
    _, kc, U, W, G, _, n = _prepare(np.zeros_like(k), k, v, g, beta, C, 1.0)
    M = np.eye(K)
    N = np.zeros((K, V))
    for c in range(n):
        decay_k = kc[c] * np.exp(G[c, -1] - G[c])[:, None]
        Mi = np.exp(G[c, -1]) * np.eye(K) - decay_k.T @ W[c]
        Ni = decay_k.T @ U[c]
        N = Mi @ N + Ni
        M = Mi @ M
    return M, N
