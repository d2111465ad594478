"""GPU parity of the whole path (gdn_shard_fwd) on P virtual shards.

Every case is compared with the unsharded fp64 oracle (conv + SiLU, L2 norm,
token recurrence) and with the GPU's own P = 1 result; the first 64 tokens
after every shard boundary and the final states are checked separately, and
long-memory gate variants make the carried state visible.  The full-size
workloads are checked on sampled (value head, state column) chains, which
the oracle computes alone.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from tests.parity import assert_close, dev, f64, path_inputs, rel_l2

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    from linear_attention_sequence_device_gb300 import build
    build.build_library()
    import linear_attention_sequence_device_gb300 as g
    g.load()
    return g


def run_gpu(w, d, P, workspace=None):
    import linear_attention_sequence_device_gb300 as g
    return g.gdn_shard_fwd(d["x"], d["conv_w"], d["conv_b"], d["g"], d["beta"], d["cu"], w.Hk,
                           w.Hv, w.dk, w.dv, P, h0=d["h0"], want_plan=True, workspace=workspace)


def oracle_path(w, host):
    return oracle.path_forward(W.as_f64(host["x"], w.dtype), host["conv_w"], host["conv_b"],
                               host["g"], host["beta"], host["h0"], w.cu_seqlens(), w.Hk, w.Hv,
                               w.dk, w.dv, w.scale)


def reduced(name, **kw):
    """Small versions of the workloads: same heads, head size, dtype and gate
    recipe; T cut down so that the oracle finishes in seconds."""
    if name == "tiny":
        return W.tiny(**kw)
    if name == "packed_varlen":
        T = 4096
        return W.Workload("packed_small", T, 16, 32, 128, 128, "bf16", kw.pop("n_shards", 1), 1,
                          W.lengths_uniform(1, T, 64, 1024), **kw)
    if name == "long":
        return W.long_seq(T=4096, **kw)
    if name == "ragged":
        T = 4096
        return W.Workload("ragged_small", T, 16, 16, 128, 128, "bf16", kw.pop("n_shards", 16), 3,
                          W.lengths_geometric(3, T, 1.0 / 300.0, 1, 4096), **kw)
    if name == "million":
        return W.million(T=4096, **kw)
    raise KeyError(name)


CASES = [
    ("tiny", {}), ("tiny", {"n_shards": 8}), ("tiny", {"n_shards": 1}),
    ("tiny", {"g_shift": -4.0}), ("tiny", {"g_zero": True, "n_shards": 4}),
    ("packed_varlen", {}), ("packed_varlen", {"n_shards": 4}),
    ("long", {}), ("long", {"g_shift": -4.0}), ("long", {"g_zero": True}),
    ("ragged", {}), ("ragged", {"g_shift": -4.0, "n_shards": 8}),
    ("million", {}), ("million", {"g_shift": -6.0}), ("million", {"g_zero": True, "n_shards": 16}),
]


@pytest.mark.parametrize("name,kw", CASES, ids=lambda c: str(c))
def test_shard_fwd_vs_oracle(name, kw):
    w = reduced(name, **kw)
    host, d = path_inputs(w)
    o, hf, plan = run_gpu(w, d, w.n_shards)
    o_ref, hf_ref = oracle_path(w, host)
    assert_close(f64(o), o_ref, w.dtype, "o")
    assert_close(f64(hf), hf_ref, w.dtype, "h_final")
    # the plan the path used is the oracle's plan
    import linear_attention_sequence_device_gb300 as g
    status, recs = g.decode_plan(plan, w.N, w.n_shards)
    assert status == 0
    for a, b in zip(recs, oracle.plan(w.cu_seqlens(), w.n_shards)):
        assert a["local_cu"] == b["local_cu"].tolist()
        assert a["pre_num_conv_tokens"] == b["pre_num_conv_tokens"]
    # the first chunk after every shard boundary, where carried state matters most
    part = w.T // w.n_shards
    of, orf = f64(o), o_ref
    for r in range(1, w.n_shards):
        sl = slice(r * part, min(r * part + 64, w.T))
        assert_close(of[sl], orf[sl], w.dtype, f"o after boundary {r}")
    # sharded == unsharded on the GPU
    if w.n_shards > 1:
        o1, hf1, _ = run_gpu(w, d, 1)
        assert_close(f64(o), f64(o1), w.dtype, "o (P vs 1)")
        assert_close(f64(hf), f64(hf1), w.dtype, "h_final (P vs 1)")


def test_long_memory_state_is_carried():
    """With g = 0 the state never decays, so dropping the carried state is a
    first-order error: the sharded path matches the oracle, while the
    oracle's own restart-from-zero at every shard boundary (the negative
    control) misses the bar by far after the first boundary."""
    w = reduced("long", g_zero=True)
    host, d = path_inputs(w)
    P = 8
    o, hf, _ = run_gpu(w, d, P)
    o_ref, hf_ref = oracle_path(w, host)
    assert_close(f64(o), o_ref, w.dtype, "o")
    assert_close(f64(hf), hf_ref, w.dtype, "h_final")
    # negative control: every shard restarted from a zero state
    part = w.T // P
    cu = np.arange(0, w.T + 1, part, dtype=np.int64)
    o_restart, _ = oracle.path_forward(W.as_f64(host["x"], w.dtype), host["conv_w"], host["conv_b"], host["g"],
                                       host["beta"], None, cu, w.Hk, w.Hv, w.dk, w.dv, w.scale)
    for r in range(1, P):
        sl = slice(r * part, (r + 1) * part)
        assert rel_l2(f64(o)[sl], o_ref[sl]) < 1e-2
        assert rel_l2(o_restart[sl], o_ref[sl]) > 0.1, r


def test_sharded_conv_is_bit_identical():
    """The conv that reads its halo from the previous shard's rows equals the
    unsharded conv bit for bit (conv output sits after the plan in the workspace)."""
    import linear_attention_sequence_device_gb300 as g
    w = reduced("ragged")
    _, d = path_inputs(w)
    outs = []
    for P in (1, 16):
        ws = torch.empty(g.shard_fwd_workspace_size(w.T, w.N, P, w.Hk, w.Hv, w.dk, w.dv,
                                                    torch.bfloat16), dtype=torch.uint8, device=dev())
        run_gpu(w, d, P, workspace=ws)
        off = (4 * g.plan_words(w.N, P) + 255) // 256 * 256
        outs.append(ws[off:off + w.T * w.Cch * 2].clone())
    assert torch.equal(outs[0], outs[1])


def test_bad_cu_seqlens_leaves_outputs_untouched():
    import linear_attention_sequence_device_gb300 as g
    w = reduced("tiny")
    _, d = path_inputs(w)
    d["cu"] = torch.tensor([0, 200, 100, 256], dtype=torch.int32, device=dev())
    o = torch.full((w.T, w.Hv, w.dv), 7.0, device=dev())
    _, _, plan = g.gdn_shard_fwd(d["x"], d["conv_w"], None, d["g"], d["beta"], d["cu"], w.Hk,
                                 w.Hv, w.dk, w.dv, 2, out=o, want_plan=True)
    torch.cuda.synchronize()
    assert int(plan[0]) == 6
    assert bool((o == 7.0).all())


# ---------------------------------------------------------------------------
# full-size workloads, sampled chains
# ---------------------------------------------------------------------------

def sampled_oracle(w, heads, cols):
    """Oracle output for value heads `heads`, state columns `cols`, all tokens:
    conv of just the needed channels, then the token recurrence."""
    G = w.Hv // w.Hk
    out = {}
    cu = w.cu_seqlens()
    cw = W.as_f64(w.conv_w(), w.dtype)
    g_all = w.g()
    b_all = W.as_f64(w.beta(), w.dtype)
    h0 = w.h0()
    for h in heads:
        hk = h // G
        chans = (list(range(hk * w.dk, (hk + 1) * w.dk))
                 + list(range(w.Hk * w.dk + hk * w.dk, w.Hk * w.dk + (hk + 1) * w.dk))
                 + [2 * w.Hk * w.dk + h * w.dv + c for c in cols])
        xs = _gather_cols(w, chans)
        y = oracle.conv_silu(xs, cw[chans], None, cu)
        q = y[:, :w.dk].reshape(w.T, 1, w.dk)
        k = y[:, w.dk:2 * w.dk].reshape(w.T, 1, w.dk)
        v = y[:, 2 * w.dk:].reshape(w.T, 1, len(cols))
        hh = None if h0 is None else h0[:, h:h + 1][..., cols].astype(np.float64)
        o, hf = oracle.gdn_forward(q, k, v, g_all[:, h:h + 1].astype(np.float64), b_all[:, h:h + 1],
                                   hh, cu, w.scale, l2norm=True)
        out[h] = (o[:, 0], hf[:, 0])
    return out


def _gather_cols(w, chans):
    """Generate only the needed channels (contiguous runs) of the raw input."""
    runs, start = [], chans[0]
    prev = start
    for c in chans[1:] + [None]:
        if c is None or c != prev + 1:
            runs.append((start, prev + 1))
            if c is not None:
                start = c
        if c is not None:
            prev = c
    parts = [W.as_f64(w.x(cols=r), w.dtype) for r in runs]
    return np.concatenate(parts, axis=1)


FULL = ["packed_varlen", "long", "ragged", "million"]


def _spread(n, k):
    """k indices spread over range(n), both ends included."""
    return sorted({int(round(i * (n - 1) / (k - 1))) for i in range(k)})


@pytest.mark.parametrize("name", FULL)
def test_full_size_sampled(name):
    """Full-size workloads at their own shard counts: four value heads spread
    over the range and eight state columns in every 32-column piece, all
    tokens and the final states; on the single-sequence workloads also the
    first 64 tokens after every shard boundary on their own."""
    w = W.CONFIGS[name]()
    _, d = path_inputs(w)
    o, hf, _ = run_gpu(w, d, w.n_shards)
    heads = _spread(w.Hv, 4)
    cols = sorted({p * 32 + c for p in range(w.dv // 32) for c in (0, 3, 7, 12, 18, 23, 27, 31)})
    ref = sampled_oracle(w, heads, cols)
    part = w.T // w.n_shards
    for h in heads:
        o_ref, hf_ref = ref[h]
        og = f64(o[:, h, cols])
        assert_close(og, o_ref, w.dtype, f"{name} o head {h}")
        assert_close(f64(hf[:, h][..., cols]), hf_ref, w.dtype, f"{name} h_final head {h}")
        if w.N == 1:
            for r in range(1, w.n_shards):
                sl = slice(r * part, r * part + 64)
                assert_close(og[sl], o_ref[sl], w.dtype, f"{name} o head {h} after boundary {r}")
    del d, o, hf
    torch.cuda.empty_cache()


@pytest.mark.parametrize("name,P,kw", [("long", 8, {}), ("long", 4, {"g_zero": True}), ("ragged", 16, {}),
                                       ("million", 16, {}), ("long_ragged_tail", 8, {})])
def test_summary_m_chains_apart_are_bit_identical(name, P, kw):
    """With the full workspace the summaries' M halves run in their own kernel
    from the W rows, K~ tiles and e^{G_last} that the N halves stored; with the
    minimum workspace they run in the chunk kernel.  Both compute the same
    products on the same operands, so o and h_final agree bit for bit."""
    import linear_attention_sequence_device_gb300 as g
    if name == "long_ragged_tail":  # shards of 500 tokens: a partial last chunk in every shard
        w = W.long_seq(T=4000, n_shards=P, h0_std=0.02)
    else:
        w = reduced(name, n_shards=P, **kw)
    host, d = path_inputs(w)
    dt = torch.bfloat16
    full = g.shard_fwd_workspace_size(w.T, w.N, P, w.Hk, w.Hv, w.dk, w.dv, dt)
    small = g.shard_fwd_workspace_min_size(w.T, w.N, P, w.Hk, w.Hv, w.dk, w.dv, dt)
    assert full > small > 0
    g.binding.device_timeouts(reset=True)
    o1, hf1, plan1 = run_gpu(w, d, P, workspace=torch.empty(full, dtype=torch.uint8, device=dev()))
    o2, hf2, plan2 = run_gpu(w, d, P, workspace=torch.empty(small, dtype=torch.uint8, device=dev()))
    torch.cuda.synchronize()
    assert int(plan1[0]) == 0 and int(plan2[0]) == 0
    assert torch.equal(o1, o2)
    assert torch.equal(hf1, hf2)
    assert g.binding.device_timeouts() == 0
    if name == "long_ragged_tail":  # and the result is the oracle's
        o_ref, hf_ref = oracle_path(w, host)
        assert_close(f64(o1), o_ref, w.dtype, "o")
        assert_close(f64(hf1), hf_ref, w.dtype, "h_final")
