"""Pins of the fp64 oracle against things other than itself (CPU only).

Plan    : hand-enumerated cases (tests/golden/plan_cases.json), a brute-force
          per-token derivation on random inputs, and structural invariants.
Conv    : torch.nn.functional.conv1d (the non-sharded path of the
          hyper-parallel page), zero-halo equivalence, a K=1 special case.
GDN     : the chunked WY/UT form restated independently in numpy, closed
          forms (beta = 0, d = 1, orthonormal keys), linearity, the sharding
          identity through explicit K x K matrix products, resume.
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle
from tests import chunk_form_np as cf

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
rng = np.random.default_rng(1234)


# ----------------------------------------------------------------------------
# plan
# ----------------------------------------------------------------------------

def test_plan_hand_cases():
    cases = json.load(open(os.path.join(GOLDEN, "plan_cases.json")))["cases"]
    for case in cases:
        got = oracle.plan(case["cu"], case["P"])
        for r, exp in enumerate(case["shards"]):
            rec = got[r]
            assert rec["local_cu"].tolist() == exp[0], (case["name"], r)
            assert rec["pre_num_ranks"] == exp[1], (case["name"], r)
            assert rec["is_first_rank"] == exp[2], (case["name"], r)
            assert rec["post_num_ranks"] == exp[3], (case["name"], r)
            assert rec["is_last_rank"] == exp[4], (case["name"], r)
            assert rec["pre_num_conv_tokens"] == exp[5], (case["name"], r)
            assert rec["start_seq_idx"] == exp[6], (case["name"], r)


def brute_plan(cu, P):
    """Re-derive every plan field from a per-token (owner shard, sequence) table."""
    cu = np.asarray(cu)
    T = int(cu[-1])
    part = T // P
    sid = np.empty(T, dtype=np.int64)
    for i in range(len(cu) - 1):
        sid[cu[i]:cu[i + 1]] = i
    owner = np.arange(T) // part
    out = []
    for r in range(P):
        rs, re = r * part, (r + 1) * part
        local = [0] + [t - rs for t in range(rs + 1, re) if sid[t] != sid[t - 1]] + [part]
        seqs = [int(sid[rs + b]) for b in local[:-1]]  # owner sequence of each segment's first token
        first_seq, last_seq = sid[rs], sid[re - 1]
        first_tok = np.flatnonzero(sid == first_seq)[0]
        last_tok = np.flatnonzero(sid == last_seq)[-1]
        out.append(dict(local_cu=local, local_seq=seqs,
                        start_seq_idx=int(first_seq),
                        pre_num_conv_tokens=int(np.sum(sid[:rs] == first_seq)),
                        pre_num_ranks=int(r - owner[first_tok]),
                        post_num_ranks=int(owner[last_tok] - r),
                        is_first_rank=int(owner[first_tok] == r),
                        is_last_rank=int(owner[last_tok] == r)))
    return out


@pytest.mark.parametrize("trial", range(300))
def test_plan_brute_force(trial):
    r = np.random.default_rng(trial)
    P = int(r.choice([1, 2, 3, 4, 5, 8]))
    part = int(r.integers(1, 12))
    T = P * part
    # random lengths incl. empty sequences, summing to T
    cuts = np.sort(r.integers(0, T + 1, size=int(r.integers(0, 8))))
    cu = np.concatenate([[0], cuts, [T]]).astype(np.int64)
    got = oracle.plan(cu, P)
    exp = brute_plan(cu, P)
    for a, b in zip(got, exp):
        assert a["local_cu"].tolist() == b["local_cu"]
        assert a["local_seq"].tolist() == b["local_seq"]
        for f in ("start_seq_idx", "pre_num_conv_tokens", "pre_num_ranks", "post_num_ranks",
                  "is_first_rank", "is_last_rank"):
            assert a[f] == b[f], f


@pytest.mark.parametrize("trial", range(50))
def test_plan_invariants(trial):
    r = np.random.default_rng(10_000 + trial)
    P = int(r.choice([2, 4, 8, 16]))
    part = int(r.integers(1, 40))
    T = P * part
    lens = r.integers(1, 3 * part + 2, size=64)
    cu = np.concatenate([[0], np.cumsum(lens)])
    cu = np.unique(np.minimum(cu, T))
    got = oracle.plan(cu, P)
    # concatenating local boundaries reproduces the clamped global boundaries
    glob = sorted({0} | {rec["local_cu"][i] + r_ * part for r_, rec in enumerate(got)
                         for i in range(len(rec["local_cu"]))})
    assert glob == sorted(set(np.clip(cu, 0, T).tolist()) | {p * part for p in range(P + 1)})
    for r_, rec in enumerate(got):
        assert rec["local_cu"][0] == 0 and rec["local_cu"][-1] == part
        if r_ > 0:
            assert (not rec["is_first_rank"]) == (got[r_ - 1]["post_num_ranks"] >= 1)
            if len(got[r_ - 1]["local_cu"]) == 2 and not got[r_ - 1]["is_first_rank"]:
                # previous shard spanned entirely by one sequence
                if not rec["is_first_rank"]:
                    assert rec["pre_num_ranks"] == got[r_ - 1]["pre_num_ranks"] + 1


# ----------------------------------------------------------------------------
# conv
# ----------------------------------------------------------------------------

def torch_conv_silu(x, w, b, cu):
    """Per sequence: conv1d(padding=K-1)[..., :len] then SiLU (library routine)."""
    C, Kc = w.shape
    out = np.zeros_like(x)
    for i in range(len(cu) - 1):
        s0, s1 = cu[i], cu[i + 1]
        if s1 == s0:
            continue
        xt = torch.from_numpy(x[s0:s1].T.copy())[None]          # [1, C, L]
        y = torch.nn.functional.conv1d(xt, torch.from_numpy(w.copy())[:, None, :],
                                       None if b is None else torch.from_numpy(b.copy()),
                                       padding=Kc - 1, groups=C)[0, :, : s1 - s0]
        out[s0:s1] = torch.nn.functional.silu(y).T.numpy()
    return out


@pytest.mark.parametrize("Kc", [1, 2, 3, 4])
@pytest.mark.parametrize("bias", [False, True])
def test_conv_vs_torch(Kc, bias):
    T, C = 97, 24
    x = rng.standard_normal((T, C))
    w = rng.standard_normal((C, Kc)) * 0.5
    b = rng.standard_normal(C) if bias else None
    cu = np.array([0, 1, 4, 40, 40, 97])
    np.testing.assert_allclose(oracle.conv_silu(x, w, b, cu), torch_conv_silu(x, w, b, cu),
                               rtol=1e-12, atol=1e-12)


def test_conv_halo_equals_concatenation():
    T, C, Kc = 50, 16, 4
    x = rng.standard_normal((T, C))
    w = rng.standard_normal((C, Kc))
    for split in (3, 7, 20):
        full = oracle.conv_silu(x, w, None, [0, T])
        halo = x[split - (Kc - 1):split]
        part = oracle.conv_silu(x[split:], w, None, [0, T - split], halo=halo, halo_len=Kc - 1)
        np.testing.assert_array_equal(part, full[split:])
    # zero-length halo = fresh sequence
    np.testing.assert_array_equal(
        oracle.conv_silu(x[10:], w, None, [0, T - 10], halo=np.ones((Kc - 1, C)), halo_len=0),
        oracle.conv_silu(x[10:], w, None, [0, T - 10]))
    # partial halo: only the last 2 rows are real history
    h2 = oracle.conv_silu(x[10:], w, None, [0, T - 10], halo=x[7:10], halo_len=2)
    np.testing.assert_array_equal(h2, oracle.conv_silu(x[8:], w, None, [0, T - 8])[2:])


def test_conv_k1_identity():
    x = rng.standard_normal((30, 8))
    b = rng.standard_normal(8)
    y = oracle.conv_silu(x, np.ones((8, 1)), b, [0, 30])
    z = x + b
    np.testing.assert_allclose(y, z / (1 + np.exp(-z)), rtol=1e-15)


# ----------------------------------------------------------------------------
# gated delta rule
# ----------------------------------------------------------------------------

def rand_inputs(T, Hk, Hv, K, V, r=rng, unit=True, g_scale=1.0):
    q = r.standard_normal((T, Hk, K))
    k = r.standard_normal((T, Hk, K))
    if unit:
        q /= np.linalg.norm(q, axis=-1, keepdims=True)
        k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = r.standard_normal((T, Hv, V))
    g = -np.log1p(np.exp(r.standard_normal((T, Hv)))) * g_scale
    beta = 1 / (1 + np.exp(-r.standard_normal((T, Hv))))
    return q, k, v, g, beta


@pytest.mark.parametrize("L", [1, 63, 64, 65, 200])
def test_gdn_vs_chunk_form(L):
    K, V = 16, 8
    q, k, v, g, beta = rand_inputs(L, 1, 1, K, V)
    h0 = rng.standard_normal((1, 1, K, V)) * 0.3
    o, hf = oracle.gdn_forward(q, k, v, g, beta, h0, [0, L], K ** -0.5)
    o2, S2 = cf.chunk_forward(q[:, 0], k[:, 0], v[:, 0], g[:, 0], beta[:, 0], h0[0, 0])
    np.testing.assert_allclose(o[:, 0], o2, rtol=0, atol=1e-12)
    np.testing.assert_allclose(hf[0, 0], S2, rtol=0, atol=1e-12)
    M, N = cf.chunk_summary(k[:, 0], v[:, 0], g[:, 0], beta[:, 0])
    Mo, No = oracle.gdn_summary(k, v, g, beta, [0, L])
    np.testing.assert_allclose(Mo[0, 0], M, atol=1e-12)
    np.testing.assert_allclose(No[0, 0], N, atol=1e-12)


def test_gdn_chunk_form_long_memory_and_gqa():
    T, Hk, Hv, K, V = 150, 2, 4, 8, 8
    q, k, v, g, beta = rand_inputs(T, Hk, Hv, K, V, g_scale=0.01)
    cu = [0, 70, 70, 150]
    o, hf = oracle.gdn_forward(q, k, v, g, beta, None, cu, 0.37)
    for n in range(3):
        s0, s1 = cu[n], cu[n + 1]
        for h in range(Hv):
            hk = h // (Hv // Hk)
            if s1 == s0:
                np.testing.assert_array_equal(hf[n, h], 0)
                continue
            o2, S2 = cf.chunk_forward(q[s0:s1, hk], k[s0:s1, hk], v[s0:s1, h], g[s0:s1, h],
                                      beta[s0:s1, h], None, scale=0.37)
            np.testing.assert_allclose(o[s0:s1, h], o2, atol=1e-11)
            np.testing.assert_allclose(hf[n, h], S2, atol=1e-11)


def test_beta_zero_is_pure_decay():
    T, K, V = 40, 8, 6
    q, k, v, g, _ = rand_inputs(T, 1, 1, K, V)
    h0 = rng.standard_normal((1, 1, K, V))
    o, hf = oracle.gdn_forward(q, k, v, g, np.zeros((T, 1)), h0, [0, T], 0.5)
    np.testing.assert_allclose(hf[0, 0], np.exp(g[:, 0].sum()) * h0[0, 0], rtol=1e-13)
    decay = np.exp(np.cumsum(g[:, 0]))
    np.testing.assert_allclose(o[:, 0], decay[:, None] * (0.5 * q[:, 0] @ h0[0, 0]), rtol=1e-12,
                               atol=1e-14)


def test_scalar_case():
    T = 25
    q, k, v, g, beta = rand_inputs(T, 1, 1, 1, 1, unit=False)
    o, hf = oracle.gdn_forward(q, k, v, g, beta, None, [0, T], 1.0)
    s = 0.0
    for t in range(T):
        a, b, kk = np.exp(g[t, 0]), beta[t, 0], k[t, 0, 0]
        s = a * s * (1 - b * kk * kk) + b * kk * v[t, 0, 0]
        assert abs(o[t, 0, 0] - s * q[t, 0, 0]) <= 1e-14 * (1 + abs(s))
    assert abs(hf[0, 0, 0, 0] - s) <= 1e-14


def test_orthonormal_keys_overwrite_rows():
    K, V, T = 8, 5, 20
    k = np.zeros((T, 1, K))
    k[np.arange(T), 0, np.arange(T) % K] = 1.0
    q = k.copy()
    v = rng.standard_normal((T, 1, V))
    h0 = rng.standard_normal((1, 1, K, V))
    o, hf = oracle.gdn_forward(q, k, v, np.zeros((T, 1)), np.ones((T, 1)), h0, [0, T], 1.0)
    exp = h0[0, 0].copy()
    for t in range(T):
        exp[t % K] = v[t, 0]
        # S[row] + (v - S[row]) equals v up to one rounding
        np.testing.assert_allclose(o[t, 0], v[t, 0], rtol=0, atol=1e-15 * 8)
    np.testing.assert_allclose(hf[0, 0], exp, rtol=0, atol=1e-15 * 8)


def test_linearity_in_v_and_h0():
    T, K, V = 90, 8, 4
    q, k, v1, g, beta = rand_inputs(T, 1, 1, K, V)
    v2 = rng.standard_normal(v1.shape)
    a1, a2 = rng.standard_normal((1, 1, K, V)), rng.standard_normal((1, 1, K, V))
    cu = [0, T]
    o1, s1 = oracle.gdn_forward(q, k, v1, g, beta, a1, cu, 0.3)
    o2, s2 = oracle.gdn_forward(q, k, v2, g, beta, a2, cu, 0.3)
    o3, s3 = oracle.gdn_forward(q, k, 2 * v1 - 3 * v2, g, beta, 2 * a1 - 3 * a2, cu, 0.3)
    np.testing.assert_allclose(o3, 2 * o1 - 3 * o2, atol=1e-12)
    np.testing.assert_allclose(s3, 2 * s1 - 3 * s2, atol=1e-12)


@pytest.mark.parametrize("P", [2, 4, 5])
def test_sharding_identity_explicit_products(P):
    """M_r as explicit products of K x K matrices, N_r from a zero state; the
    composed carries reproduce the unsharded state and outputs."""
    K, V, part = 6, 5, 23
    T = P * part
    q, k, v, g, beta = rand_inputs(T, 1, 1, K, V, g_scale=0.05)
    h0 = rng.standard_normal((1, 1, K, V))
    o_ref, hf_ref = oracle.gdn_forward(q, k, v, g, beta, h0, [0, T], 0.4)
    Ms, Ns = [], []
    for r in range(P):
        sl = slice(r * part, (r + 1) * part)
        M = np.eye(K)
        for t in range(r * part, (r + 1) * part):
            kt = k[t, 0][:, None]
            M = (np.exp(g[t, 0]) * (np.eye(K) - beta[t, 0] * kt @ kt.T)) @ M
        _, N = oracle.gdn_forward(q[sl], k[sl], v[sl], g[sl], beta[sl], None, [0, part], 0.4,
                                  want_o=False)
        Mo, No = oracle.gdn_summary(k[sl], v[sl], g[sl], beta[sl], [0, part])
        np.testing.assert_allclose(Mo[0, 0], M, atol=1e-13)
        np.testing.assert_allclose(No[0, 0], N[0, 0], atol=1e-13)
        Ms.append(M)
        Ns.append(N[0, 0])
    S_in = oracle.state_combine(np.array(Ms)[:, None], np.array(Ns)[:, None], h0[0])
    state = h0[0, 0]
    for r in range(P):
        np.testing.assert_allclose(S_in[r, 0], state, atol=1e-12)
        sl = slice(r * part, (r + 1) * part)
        o_r, s_r = oracle.gdn_forward(q[sl], k[sl], v[sl], g[sl], beta[sl], state[None, None],
                                      [0, part], 0.4)
        np.testing.assert_allclose(o_r, o_ref[sl], atol=1e-12)
        state = s_r[0, 0]
        np.testing.assert_allclose(Ms[r] @ S_in[r, 0] + Ns[r], state, atol=1e-12)
    np.testing.assert_allclose(state, hf_ref[0, 0], atol=1e-12)


def test_resume_equals_one_call():
    T, K, V = 130, 8, 8
    q, k, v, g, beta = rand_inputs(T, 2, 2, K, V)
    o, hf = oracle.gdn_forward(q, k, v, g, beta, None, [0, T], 0.35)
    o1, h1 = oracle.gdn_forward(q[:77], k[:77], v[:77], g[:77], beta[:77], None, [0, 77], 0.35)
    o2, h2 = oracle.gdn_forward(q[77:], k[77:], v[77:], g[77:], beta[77:], h1, [0, T - 77], 0.35)
    np.testing.assert_allclose(np.concatenate([o1, o2]), o, atol=1e-13)
    np.testing.assert_allclose(h2, hf, atol=1e-13)


def test_l2norm_applied_to_q_and_k():
    """With the L2-norm flag, rescaling q or k (far above the 1e-6 epsilon)
    leaves the result unchanged; without it, it does not."""
    T, K, V = 50, 8, 4
    q, k, v, g, beta = rand_inputs(T, 1, 1, K, V, unit=False)
    a = oracle.gdn_forward(q, k, v, g, beta, None, [0, T], 0.3, l2norm=True)
    b = oracle.gdn_forward(7.0 * q, 0.25 * k, v, g, beta, None, [0, T], 0.3, l2norm=True)
    # the epsilon moves the result by O(1e-6 / |x|^2); a missing norm moves it by O(1)
    np.testing.assert_allclose(b[0], a[0], rtol=0, atol=1e-5)
    np.testing.assert_allclose(b[1], a[1], rtol=0, atol=1e-5)
    c = oracle.gdn_forward(q, 0.25 * k, v, g, beta, None, [0, T], 0.3, l2norm=False)
    assert np.abs(c[0] - a[0]).max() > 1e-3
    # the normalised key has norm 1 / sqrt(1 + 1e-6 / |k|^2): unit keys stay put
    ku = k / np.linalg.norm(k, axis=-1, keepdims=True)
    qu = q / np.linalg.norm(q, axis=-1, keepdims=True)
    d = oracle.gdn_forward(qu, ku, v, g, beta, None, [0, T], 0.3, l2norm=False)
    np.testing.assert_allclose(d[0], a[0], rtol=0, atol=1e-5)
    Ms, _ = oracle.gdn_summary(k, v, g, beta, [0, T], l2norm=True)
    Mu, _ = oracle.gdn_summary(ku, v, g, beta, [0, T], l2norm=False)
    np.testing.assert_allclose(Ms, Mu, rtol=0, atol=1e-5)


def test_path_forward_composition():
    """The whole-path oracle equals conv -> split -> normalise -> recurrence."""
    T, Hk, Hv, K, V, Kc = 70, 1, 2, 8, 4, 4
    C = 2 * Hk * K + Hv * V
    x = rng.standard_normal((T, C))
    w = rng.standard_normal((C, Kc)) * 0.5
    g = -np.log1p(np.exp(rng.standard_normal((T, Hv))))
    beta = 1 / (1 + np.exp(-rng.standard_normal((T, Hv))))
    cu = [0, 33, 70]
    o, hf = oracle.path_forward(x, w, None, g, beta, None, cu, Hk, Hv, K, V, 0.3)
    y = torch_conv_silu(x, w, None, np.array(cu))
    qn = y[:, :K] / np.sqrt((y[:, :K] ** 2).sum(-1, keepdims=True) + 1e-6)
    kn = y[:, K:2 * K] / np.sqrt((y[:, K:2 * K] ** 2).sum(-1, keepdims=True) + 1e-6)
    for n in range(2):
        s0, s1 = cu[n], cu[n + 1]
        for h in range(Hv):
            o2, S2 = cf.chunk_forward(qn[s0:s1], kn[s0:s1], y[s0:s1, 2 * K + h * V:2 * K + (h + 1) * V],
                                      g[s0:s1, h], beta[s0:s1, h], None, scale=0.3)
            np.testing.assert_allclose(o[s0:s1, h], o2, atol=1e-11)
            np.testing.assert_allclose(hf[n, h], S2, atol=1e-11)


# ----------------------------------------------------------------------------
# gates from the raw projections and the gated RMS norm (the wrappers'
# forward around the path)
# ----------------------------------------------------------------------------

def test_gates_closed_forms():
    """a = -dt_bias gives softplus(0) = ln 2, so g = -exp(A_log) ln 2; b = 0
    gives beta = 1/2; A_log = log 3 scales the decay rate by exactly 3."""
    T, Hv = 5, 4
    dt = rng.standard_normal(Hv)
    A_log = rng.standard_normal(Hv)
    g, beta = oracle.gates(-np.tile(dt, (T, 1)), np.zeros((T, Hv)), A_log, dt)
    np.testing.assert_allclose(g, -np.exp(A_log)[None, :] * np.log(2.0) * np.ones((T, 1)), rtol=1e-15)
    np.testing.assert_allclose(beta, 0.5, rtol=0)
    a = rng.standard_normal((T, Hv))
    g1, _ = oracle.gates(a, a, np.zeros(Hv), dt)
    g3, _ = oracle.gates(a, a, np.full(Hv, np.log(3.0)), dt)
    np.testing.assert_allclose(g3, 3.0 * g1, rtol=1e-14)
    assert (g1 < 0).all()


def test_gates_vs_torch():
    """Against torch's softplus (threshold 20: identical up to e^-20 beyond
    it) and sigmoid, over a wide range of inputs."""
    T, Hv = 200, 6
    a = rng.standard_normal((T, Hv)) * 8.0
    b = rng.standard_normal((T, Hv)) * 8.0
    A_log = rng.standard_normal(Hv)
    dt = rng.standard_normal(Hv)
    g, beta = oracle.gates(a, b, A_log, dt)
    ta = torch.tensor(a, dtype=torch.float64)
    exp_g = -torch.tensor(A_log).exp() * torch.nn.functional.softplus(ta + torch.tensor(dt))
    np.testing.assert_allclose(g, exp_g.numpy(), rtol=1e-12, atol=1e-8)
    np.testing.assert_allclose(beta, torch.sigmoid(torch.tensor(b)).numpy(), rtol=1e-13, atol=0)


def test_gated_rmsnorm_vs_torch():
    """Against torch.nn.functional.rms_norm over head_v_dim times silu(z)."""
    o = rng.standard_normal((7, 3, 128))
    z = rng.standard_normal((7, 3, 128)) * 3.0
    w = 1.0 + 0.1 * rng.standard_normal(128)
    for eps in (1e-6, 0.5):
        y = oracle.gated_rmsnorm(o, z, w, eps)
        exp = torch.nn.functional.rms_norm(torch.tensor(o), (128,), torch.tensor(w), eps) \
            * torch.nn.functional.silu(torch.tensor(z))
        np.testing.assert_allclose(y, exp.numpy(), rtol=1e-12, atol=1e-14)


def test_gated_rmsnorm_closed_forms():
    """z = 0 closes the gate (y = 0); with eps = 0 the result does not depend
    on the scale of o; a constant row c with unit weight gives silu(z)."""
    o = rng.standard_normal((4, 64))
    z = rng.standard_normal((4, 64))
    w = rng.standard_normal(64)
    assert np.all(oracle.gated_rmsnorm(o, np.zeros_like(z), w) == 0.0)
    np.testing.assert_allclose(oracle.gated_rmsnorm(37.0 * o, z, w, 0.0), oracle.gated_rmsnorm(o, z, w, 0.0),
                               rtol=1e-13)
    y = oracle.gated_rmsnorm(np.full((2, 64), 2.5), z[:2], np.ones(64), 0.0)
    np.testing.assert_allclose(y, z[:2] / (1.0 + np.exp(-z[:2])), rtol=1e-14)


# ---------------------------------------------------------------------------
# backward of the token recurrence
# ---------------------------------------------------------------------------

def _bwd_problem(seed, T_lens, Hk, Hv, K, V, h0=True):
    r = np.random.default_rng(seed)
    cu = np.concatenate([[0], np.cumsum(T_lens)]).astype(np.int64)
    T, N = int(cu[-1]), len(T_lens)
    q = r.normal(size=(T, Hk, K))
    k = r.normal(size=(T, Hk, K))
    v = r.normal(size=(T, Hv, V))
    g = -np.log1p(np.exp(r.normal(size=(T, Hv)) - 1.0))
    b = 1.0 / (1.0 + np.exp(-r.normal(size=(T, Hv))))
    h0 = r.normal(size=(N, Hv, K, V)) * 0.5 if h0 else None
    Wo = r.normal(size=(T, Hv, V))
    Wh = r.normal(size=(N, Hv, K, V))
    return cu, q, k, v, g, b, h0, Wo, Wh


@pytest.mark.parametrize("l2", [False, True])
def test_backward_vs_finite_differences(l2):
    """Every gradient against central differences of the oracle's forward
    for the loss sum(o * Wo) + sum(h_final * Wh): GQA (two value heads per
    q/k head), a 70-token sequence (two checkpointed chunks), an empty
    sequence and a short one, nonzero h0."""
    cu, q, k, v, g, b, h0, Wo, Wh = _bwd_problem(5, [70, 0, 9], 1, 2, 3, 2)
    scale = 0.7

    def loss(**a):
        o, hf = oracle.gdn_forward(a["q"], a["k"], a["v"], a["g"], a["b"], a["h0"], cu, scale,
                                   l2norm=l2)
        return float((o * Wo).sum() + (hf * Wh).sum())

    args = dict(q=q, k=k, v=v, g=g, b=b, h0=h0)
    got = oracle.gdn_backward(q, k, v, g, b, h0, cu, scale, Wo, Wh, l2norm=l2)
    names = dict(q="dq", k="dk", v="dv", g="dg", b="dbeta", h0="dh0")
    eps = 1e-6
    for nm, x in args.items():
        fd = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += eps
            xm[idx] -= eps
            fd[idx] = (loss(**{**args, nm: xp}) - loss(**{**args, nm: xm})) / (2 * eps)
        err = np.abs(fd - got[names[nm]]).max() / np.abs(fd).max()
        assert err < 1e-6, (nm, err)


def test_backward_closed_form_without_updates():
    """beta = 0: the state only decays, o_t = e^{G_t} S0^T (scale q_t), so
    dv = dk = 0, dh0 = sum_t e^{G_t} scale q_t do_t^T + e^{G_T} dh_final,
    dq_t = scale e^{G_t} S0 do_t and dbeta_t = k_t . (dS_t u_t)."""
    cu, q, k, v, g, b, h0, Wo, Wh = _bwd_problem(6, [23], 1, 1, 4, 3)
    b = np.zeros_like(b)
    scale = 0.5
    got = oracle.gdn_backward(q, k, v, g, b, h0, cu, scale, Wo, Wh)
    G = np.cumsum(g[:, 0])
    S0 = h0[0, 0]
    assert np.abs(got["dv"]).max() == 0 and np.abs(got["dk"]).max() == 0
    dh0 = np.exp(G[-1]) * Wh[0, 0] + sum(np.exp(G[t]) * scale * np.outer(q[t, 0], Wo[t, 0])
                                         for t in range(23))
    np.testing.assert_allclose(got["dh0"][0, 0], dh0, rtol=1e-12, atol=1e-12)
    dq = np.stack([scale * np.exp(G[t]) * (S0 @ Wo[t, 0]) for t in range(23)])
    np.testing.assert_allclose(got["dq"][:, 0], dq, rtol=1e-12, atol=1e-12)
    # dbeta_t = k_t^T dS_t u_t with u_t = v_t - e^{G_t} S0^T k_t and dS_t the
    # gradient w.r.t. S_t: e^{G_T - G_t} dh_final + sum_{s >= t} e^{G_s - G_t} scale q_s do_s^T
    for t in (0, 11, 22):
        dS = np.exp(G[-1] - G[t]) * Wh[0, 0] + sum(np.exp(G[s] - G[t]) * scale * np.outer(q[s, 0], Wo[s, 0])
                                                   for s in range(t, 23))
        u = v[t, 0] - np.exp(G[t]) * S0.T @ k[t, 0]
        np.testing.assert_allclose(got["dbeta"][t, 0], k[t, 0] @ dS @ u, rtol=1e-10)


def test_backward_linear_in_output_gradients():
    """The gradients are linear in (do, dh_final)."""
    cu, q, k, v, g, b, h0, Wo, Wh = _bwd_problem(7, [40, 30], 2, 4, 5, 4)
    a1 = oracle.gdn_backward(q, k, v, g, b, h0, cu, 1.0, Wo, None)
    a2 = oracle.gdn_backward(q, k, v, g, b, h0, cu, 1.0, np.zeros_like(Wo), Wh)
    a3 = oracle.gdn_backward(q, k, v, g, b, h0, cu, 1.0, 2 * Wo, -3 * Wh)
    for x in a1:
        np.testing.assert_allclose(a3[x], 2 * a1[x] - 3 * a2[x], rtol=1e-9, atol=1e-9)
