"""GPU parity of the backward of the gated delta rule (gdn_chunk_bwd, through
the C ABI) against the fp64 oracle's reverse-mode gradients.

Both sides read the same stored inputs (bf16 values where the dtype is bf16)
and the same loss gradients, so the only differences are the GPU's fp32
arithmetic and summation order: the bar is relative L2 <= 1e-4 for fp32
inputs and 1e-3 for bf16 inputs (whose sums run over up to 128 x 128 state
products of values two orders of magnitude apart), per gradient."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from tests.parity import chunk_inputs, dev, f64, rel_l2, to_dev

pytestmark = pytest.mark.gpu

TOL = {"f32": 1e-4, "bf16": 1e-3}

CASES = [
    # dtype, Hk, Hv, dk, dv, lengths, h0_std, g_shift, l2, with dh_final
    ("f32", 2, 2, 32, 32, (256,), 0.0, 0.0, False, True),
    ("f32", 1, 2, 64, 32, (100, 0, 37, 150), 0.1, -3.0, False, True),
    ("f32", 2, 2, 128, 64, (65, 130), 0.05, 0.0, True, False),
    ("bf16", 2, 4, 32, 32, (1, 63, 64, 65, 0, 300), 0.05, 0.0, False, True),
    ("bf16", 2, 4, 64, 64, (200, 129), 0.0, -4.0, True, True),
    ("bf16", 2, 2, 128, 128, (700, 33, 64), 0.02, 0.0, True, True),
    ("bf16", 1, 2, 64, 128, (257,), 0.0, 0.0, False, False),
    ("bf16", 2, 2, 128, 32, (190,), 0.1, -2.0, False, True),
    ("bf16", 2, 2, 32, 128, (99,), 0.0, 0.0, True, True),
    # strongly decaying gates, and empty sequences only around short ones
    ("bf16", 2, 2, 128, 128, (300, 77), 0.05, 4.0, False, True),
    ("bf16", 2, 2, 128, 128, (0, 130, 0, 70, 0), 0.05, 0.0, True, True),
]


def run_case(case, seed=21):
    dtype, Hk, Hv, dk, dv, lengths, h0_std, g_shift, l2, with_dh = case
    w = W.Workload("bwd", int(sum(lengths)), Hk, Hv, dk, dv, dtype, 1, seed, tuple(lengths),
                   h0_std=h0_std, g_shift=g_shift)
    host, d = chunk_inputs(w)
    if l2:  # un-normalised q, k so that the norm's backward matters
        for name in ("q", "k"):
            x = host[name] * np.linspace(0.5, 2.0, w.T)[:, None, None]
            t = torch.tensor(x, dtype=torch.float32, device=dev()).to(d[name].dtype)
            d[name] = t
            host[name] = f64(t)
    r = np.random.default_rng(seed + 1)
    do_d = torch.tensor(r.normal(size=(w.T, Hv, dv)), dtype=torch.float32, device=dev()).to(d["v"].dtype)
    dh = r.normal(size=(w.N, Hv, dk, dv)) if with_dh else None
    dh_d = None if dh is None else torch.tensor(dh, dtype=torch.float32, device=dev())
    got = __import__("linear_attention_sequence_device_gb300").gdn_chunk_bwd(
        d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu"], do_d, h0=d["h0"], dh_final=dh_d, l2norm=l2)
    torch.cuda.synchronize()
    exp = oracle.gdn_backward(host["q"], host["k"], host["v"], host["g"], host["beta"], host["h0"],
                              w.cu_seqlens(), w.scale, f64(do_d), dh, l2norm=l2)
    return w, got, exp


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"{c[0]}-{c[3]}x{c[4]}-{len(c[5])}seq-l2{int(c[8])}")
def test_chunk_bwd_vs_oracle(case):
    w, got, exp = run_case(case)
    for name in ("dq", "dk", "dv", "dg", "dbeta", "dh0"):
        r = rel_l2(f64(got[name]), exp[name])
        assert r <= TOL[w.dtype], f"{name}: relative L2 {r:.3e} > {TOL[w.dtype]}"


def test_chunk_bwd_rejects_bad_arguments():
    import linear_attention_sequence_device_gb300 as g
    lib = g.load()
    assert lib.gdn_chunk_bwd_workspace_size(64, 1, 1, 1, 48, 64) == 0
    st = lib.gdn_chunk_bwd(None, None, None, 0, 0, 0, 1, None, None, None, None, None, None, 1, 0, 1, 1,
                           128, 128, 1.0, 0, None, None, None, None, None, None, None, 0, None)
    assert st != 0  # cu_seqlens / dh0 missing


# ---------------------------------------------------------------------------
# the backward across virtual shards (gdn_shard_bwd)
# ---------------------------------------------------------------------------

# The sharded backward takes each piece's start state from the forward
# summaries, which for bf16 d = 128 run on the tensor cores with bf16 state
# operands (as the sharded forward does): its bar is the forward's, relative
# L2 <= 1e-2 for bf16, 1e-4 for fp32.
TOL_SHARD = {"f32": 1e-4, "bf16": 1e-2}

SHARD_CASES = [
    # dtype, Hk, Hv, dk, dv, lengths, h0_std, g_shift, l2, dh_final, P
    ("f32", 2, 2, 32, 32, (256,), 0.0, -4.0, False, True, 2),
    ("f32", 1, 2, 64, 32, (100, 0, 37, 119), 0.1, -4.0, False, True, 4),
    ("bf16", 2, 2, 128, 128, (2048,), 0.02, -6.0, True, True, 8),
    ("bf16", 2, 4, 64, 64, (300, 1, 0, 211, 512), 0.05, -4.0, False, True, 4),
    ("bf16", 2, 2, 128, 128, (700, 33, 64, 227), 0.02, 0.0, True, False, 4),
]


def run_shard_case(case, seed=31):
    dtype, Hk, Hv, dk, dv, lengths, h0_std, g_shift, l2, with_dh, P = case
    w = W.Workload("sbwd", int(sum(lengths)), Hk, Hv, dk, dv, dtype, P, seed, tuple(lengths),
                   h0_std=h0_std, g_shift=g_shift)
    host, d = chunk_inputs(w)
    r = np.random.default_rng(seed + 1)
    do_d = torch.tensor(r.normal(size=(w.T, Hv, dv)), dtype=torch.float32, device=dev()).to(d["v"].dtype)
    dh = r.normal(size=(w.N, Hv, dk, dv)) if with_dh else None
    dh_d = None if dh is None else torch.tensor(dh, dtype=torch.float32, device=dev())
    import linear_attention_sequence_device_gb300 as g
    got = g.gdn_chunk_bwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu"], do_d, h0=d["h0"], dh_final=dh_d,
                          l2norm=l2, n_shards=P, want_plan=True)
    ref = g.gdn_chunk_bwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu"], do_d, h0=d["h0"], dh_final=dh_d,
                          l2norm=l2)
    torch.cuda.synchronize()
    exp = oracle.gdn_backward(host["q"], host["k"], host["v"], host["g"], host["beta"], host["h0"],
                              w.cu_seqlens(), w.scale, f64(do_d), dh, l2norm=l2)
    return w, got, ref, exp, host, f64(do_d), dh


@pytest.mark.parametrize("case", SHARD_CASES, ids=lambda c: f"{c[0]}-{c[3]}x{c[4]}-{len(c[5])}seq-P{c[10]}")
def test_shard_bwd_vs_oracle_and_unsharded(case):
    """Every gradient of the P-shard backward against the oracle's unsharded
    backward, and against the GPU's unsharded backward; the plan is OK."""
    w, got, ref, exp, *_ = run_shard_case(case)
    assert int(got["plan"][0]) == 0
    for name in ("dq", "dk", "dv", "dg", "dbeta", "dh0"):
        r = rel_l2(f64(got[name]), exp[name])
        assert r <= TOL_SHARD[w.dtype], f"{name} vs oracle: relative L2 {r:.3e}"
        r = rel_l2(f64(got[name]), f64(ref[name]))
        assert r <= TOL_SHARD[w.dtype], f"{name} vs unsharded: relative L2 {r:.3e}"


def test_shard_bwd_carries_the_state_gradient_back():
    """Negative control on the long-memory case: the gradients of the first
    shard's tokens computed as if no later shard existed (its end-state
    gradient taken as 0) miss the bar, so the reverse merge is what makes the
    sharded result right."""
    case = SHARD_CASES[2]
    w, got, ref, exp, host, do, dh = run_shard_case(case)
    part = w.T // case[10]
    cu0 = np.array([0, part])
    trunc = oracle.gdn_backward(host["q"][:part], host["k"][:part], host["v"][:part], host["g"][:part],
                                host["beta"][:part], host["h0"], cu0, w.scale, do[:part], None, l2norm=True)
    for name in ("dk", "dv", "dg"):
        assert rel_l2(trunc[name], exp[name][:part]) > 10 * TOL_SHARD[w.dtype], name
        assert rel_l2(f64(got[name])[:part], exp[name][:part]) <= TOL_SHARD[w.dtype], name


def test_shard_bwd_bad_cu_seqlens_sets_status():
    """A decreasing cu_seqlens: the plan's status word says so; no fault."""
    import linear_attention_sequence_device_gb300 as g
    w = W.Workload("bad", 256, 1, 1, 32, 32, "f32", 2, 3, (128, 128))
    host, d = chunk_inputs(w)
    cu = torch.tensor([0, 200, 128, 256], dtype=torch.int32, device=dev())
    do = torch.zeros((w.T, 1, 32), dtype=torch.float32, device=dev())
    out = g.gdn_chunk_bwd(d["q"], d["k"], d["v"], d["g"], d["beta"], cu, do, n_shards=2, want_plan=True)
    torch.cuda.synchronize()
    assert int(out["plan"][0]) == 6
