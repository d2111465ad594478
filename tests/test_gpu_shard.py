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


SPLIT_CASES = {
    # one sequence, shards of 1000 tokens (a partial last chunk in each): 8 x 32
    # jobs per pass, more than the SMs, so the shard passes split every item
    # into a long first part and a short tail part
    "one_seq_P8": lambda: W.million(T=8000, n_shards=8),
    # 16 shards of 16 full chunks
    "one_seq_P16": lambda: W.million(T=16384, n_shards=16),
    # a sequence ending on a shard boundary: pass-2 segments that end their
    # sequence hand over through h_final, continuing ones through their start state
    "two_seqs_P8": lambda: W.Workload("two_seqs", 8000, 32, 32, 128, 128, "bf16", 8, 5, (5000, 3000),
                                      g_shift=2.0, h0_std=0.02),
    # one sequence per shard: pass 1 only, handed over through h_final (or,
    # without final states, run whole by the first part)
    "aligned_P8": lambda: W.Workload("aligned", 8000, 32, 32, 128, 128, "bf16", 8, 6, (1000,) * 8,
                                     g_shift=2.0, h0_std=0.02),
}


@pytest.mark.parametrize("name", sorted(SPLIT_CASES))
@pytest.mark.parametrize("final,small_ws", [(True, False), (False, False), (True, True)])
def test_split_tail_parts_are_bit_identical(name, final, small_ws):
    """The shard passes' work queue splits items into a first part and a
    short tail part when the launch has more jobs than SMs; the tail part
    starts from the first part's final state (fp32, stored and reloaded
    exactly).  So the outputs equal, bit for bit, those of the same call
    with splitting turned off, and they match the oracle.  With the minimum
    workspace the summaries' M halves run in the chunk kernel and are split
    too: their tail parts continue from the first part's M instead of the
    identity."""
    import linear_attention_sequence_device_gb300 as g
    w = SPLIT_CASES[name]()
    host, d = path_inputs(w)
    P = w.n_shards
    ws = None
    if small_ws:
        ws = torch.empty(g.shard_fwd_workspace_min_size(w.T, w.N, P, w.Hk, w.Hv, w.dk, w.dv, torch.bfloat16),
                         dtype=torch.uint8, device=dev())

    def call():
        return g.gdn_shard_fwd(d["x"], d["conv_w"], d["conv_b"], d["g"], d["beta"], d["cu"], w.Hk, w.Hv,
                               w.dk, w.dv, P, h0=d["h0"], want_plan=True, h_final=final, workspace=ws)

    g.binding.device_timeouts(reset=True)
    try:
        g.binding.debug_set_split(False)
        o0, hf0, plan0 = call()
        torch.cuda.synchronize()
    finally:
        g.binding.debug_set_split(True)
    o1, hf1, plan1 = call()
    torch.cuda.synchronize()
    assert int(plan0[0]) == 0 and int(plan1[0]) == 0
    assert g.binding.device_timeouts() == 0
    assert torch.equal(o0, o1)
    if final:
        assert torch.equal(hf0, hf1)
    else:
        assert hf0 is None and hf1 is None
    o_ref, hf_ref = oracle_path(w, host)
    assert_close(f64(o1), o_ref, w.dtype, f"{name} o")
    if final:
        assert_close(f64(hf1), hf_ref, w.dtype, f"{name} h_final")


def test_split_tail_parts_wait_for_their_first_parts():
    """The shard passes do split: with first parts that never publish their
    final state (the gdn_debug_set_handover hook) the tail parts' waits run
    out after 2 ms and the call reports GDN_ERR_TIMEOUT (7) in the plan's
    status word; with splitting turned off nothing waits and the same call
    succeeds.  Normal calls afterwards report no timeout."""
    import linear_attention_sequence_device_gb300 as g
    b = g.binding
    w = SPLIT_CASES["one_seq_P16"]()
    _, d = path_inputs(w)
    b.device_timeouts(reset=True)
    try:
        b.debug_set_handover(2_000_000, publish=False)
        _, _, plan_split = run_gpu(w, d, w.n_shards)
        torch.cuda.synchronize()
        n_split = b.device_timeouts(reset=True)
        b.debug_set_split(False)
        _, _, plan_whole = run_gpu(w, d, w.n_shards)
        torch.cuda.synchronize()
        n_whole = b.device_timeouts(reset=True)
    finally:
        b.debug_set_handover()
        b.debug_set_split(True)
    assert int(plan_split[0]) == 7 and n_split >= 1
    assert int(plan_whole[0]) == 0 and n_whole == 0
    _, _, plan = run_gpu(w, d, w.n_shards)
    torch.cuda.synchronize()
    assert int(plan[0]) == 0 and b.device_timeouts() == 0


def test_summary_m_chain_segments():
    """Few long shards: each summary's M chain is cut into segments run side
    by side (here 2 spanning shards x 16 heads, 64 chunks a shard: 4
    segments; two sequences, so the call keeps its 4 shards), each from the
    identity, and M is their ordered product in fp32.  Small beta and g = 0
    keep M far from zero, and h0 reaches the last shard only through the M
    products: without h0 the last shard's outputs move by far more than the
    tolerance.  The result matches the oracle, as does the same call with
    the M chains run whole in the chunk kernel (minimum workspace)."""
    import linear_attention_sequence_device_gb300 as g
    w = W.Workload("two_seqs_seg", 16384, 16, 16, 128, 128, "bf16", 4, 7, (16320, 64), g_zero=True, h0_std=0.5)
    host, d = path_inputs(w)
    small_beta = torch.from_numpy(host["beta"] * 0.03).to(torch.bfloat16)
    host["beta"] = small_beta.double().numpy()
    d["beta"] = small_beta.to(dev())
    P = w.n_shards
    dt = torch.bfloat16
    full = g.shard_fwd_workspace_size(w.T, w.N, P, w.Hk, w.Hv, w.dk, w.dv, dt)
    small = g.shard_fwd_workspace_min_size(w.T, w.N, P, w.Hk, w.Hv, w.dk, w.dv, dt)
    g.binding.device_timeouts(reset=True)
    o1, hf1, plan1 = run_gpu(w, d, P, workspace=torch.empty(full, dtype=torch.uint8, device=dev()))
    o2, hf2, plan2 = run_gpu(w, d, P, workspace=torch.empty(small, dtype=torch.uint8, device=dev()))
    torch.cuda.synchronize()
    assert int(plan1[0]) == 0 and int(plan2[0]) == 0
    assert g.binding.device_timeouts() == 0
    o_ref, hf_ref = oracle_path(w, host)
    last = slice((P - 1) * (w.T // P), 16320)  # the last shard's part of the first sequence
    no_h0 = dict(host, h0=np.zeros_like(host["h0"]))
    o_ref0, _ = oracle_path(w, no_h0)
    assert rel_l2(o_ref0[last], o_ref[last]) > 0.2  # the carried h0 is visible
    for o, hf, tag in ((o1, hf1, "segments"), (o2, hf2, "whole")):
        assert_close(f64(o), o_ref, w.dtype, f"{tag} o")
        assert_close(f64(o)[last], o_ref[last], w.dtype, f"{tag} o, last shard")
        assert_close(f64(hf), hf_ref, w.dtype, f"{tag} h_final")


def test_one_sequence_runs_on_finer_internal_shards():
    """One 16384-token sequence on 2, 4 or 8 shards: too few chains for the
    SMs, so every call runs on 8 internal shards of 2048 tokens (and cuts
    their 96 M chains into 2 segments).  The three calls give bit-identical
    o and h_final, each returns the plan of its own
    shard count (the oracle's, field by field), and the result matches the
    oracle with a carried state that matters (g = 0, small beta, h0)."""
    import linear_attention_sequence_device_gb300 as g
    outs = []
    for P in (2, 4, 8):
        w = W.long_seq(T=16384, n_shards=P, g_zero=True, h0_std=0.5)
        host, d = path_inputs(w)
        small_beta = torch.from_numpy(host["beta"] * 0.03).to(torch.bfloat16)
        host["beta"] = small_beta.double().numpy()
        d["beta"] = small_beta.to(dev())
        g.binding.device_timeouts(reset=True)
        o, hf, plan = run_gpu(w, d, P)
        torch.cuda.synchronize()
        assert g.binding.device_timeouts() == 0
        assert plan.numel() == g.plan_words(w.N, P)
        assert g.decode_plan(plan, w.N, P) == g.decode_plan(g.gdn_cp_plan(d["cu"], P), w.N, P)
        status, recs = g.decode_plan(plan, w.N, P)
        assert status == 0 and len(recs) == P
        for a, b in zip(recs, oracle.plan(w.cu_seqlens(), P)):
            assert a["local_cu"] == b["local_cu"].tolist()
            assert a["pre_num_conv_tokens"] == b["pre_num_conv_tokens"]
        outs.append((o, hf))
    for o, hf in outs[1:]:
        assert torch.equal(o, outs[0][0]) and torch.equal(hf, outs[0][1])
    o_ref, hf_ref = oracle_path(w, host)
    assert_close(f64(outs[0][0]), o_ref, w.dtype, "o")
    assert_close(f64(outs[0][1]), hf_ref, w.dtype, "h_final")
    for r in range(1, 8):  # the first chunk after every internal boundary
        sl = slice(r * 2048, r * 2048 + 64)
        assert_close(f64(outs[0][0])[sl], o_ref[sl], w.dtype, f"o after {r * 2048}")


def test_shard_fwd_with_empty_sequences():
    """Empty sequences at the start, inside a shard, on a shard boundary and
    at the end: every segment finds its global sequence (h0, h_final) in the
    plan's segment map, empty sequences get h_final = h0, and the result is
    the oracle's, sharded and not."""
    w = W.Workload("empty_seqs", 4096, 16, 32, 128, 128, "bf16", 4, 11, (0, 700, 0, 324, 1024, 0, 0, 2048, 0),
                   g_shift=-4.0, h0_std=0.5)
    host, d = path_inputs(w)
    o_ref, hf_ref = oracle_path(w, host)
    for P in (4, 1):
        o, hf, plan = run_gpu(w, d, P)
        torch.cuda.synchronize()
        assert int(plan[0]) == 0
        assert_close(f64(o), o_ref, w.dtype, f"o P={P}")
        assert_close(f64(hf), hf_ref, w.dtype, f"h_final P={P}")
        for n in (0, 2, 5, 6, 8):  # the empty ones keep h0 exactly
            assert torch.equal(hf[n], d["h0"][n])
