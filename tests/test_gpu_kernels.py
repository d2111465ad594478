"""GPU parity of each entry point against the fp64 oracle (through the C ABI).

plan: bit-exact.  Floats: relative L2 <= 1e-2 (bf16) / 1e-4 (fp32) and
max-abs <= 2e-2 (the stated parity bars).  Sizes span several 64-token chunks
with ragged tails, empty sequences and every supported head size.
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from tests.parity import assert_close, chunk_inputs, dev, f64, path_inputs, rel_l2, to_dev

pytestmark = pytest.mark.gpu
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="module", autouse=True)
def lib():
    from linear_attention_sequence_device_gb300 import build
    build.build_library()
    import linear_attention_sequence_device_gb300 as g
    g.load()
    return g


def gpu_plan(cu, P):
    import linear_attention_sequence_device_gb300 as g
    cu_t = torch.tensor(np.asarray(cu), dtype=torch.int32, device=dev())
    words = g.gdn_cp_plan(cu_t, P)
    return g.decode_plan(words, len(cu) - 1, P)


def compare_plan(cu, P):
    status, recs = gpu_plan(cu, P)
    assert status == 0
    exp = oracle.plan(cu, P)
    off = 0
    for r, (a, b) in enumerate(zip(recs, exp)):
        assert a["local_cu"] == b["local_cu"].tolist(), r
        assert a["local_seq"] == b["local_seq"].tolist(), r
        for f in ("start_seq_idx", "end_seq_idx", "pre_num_ranks", "post_num_ranks",
                  "is_first_rank", "is_last_rank", "pre_num_conv_tokens"):
            assert a[f] == b[f], (r, f, a[f], b[f])
        assert a["local_num_seqs"] == len(b["local_cu"]) - 1
        assert a["seg_offset"] == off
        off += a["local_num_seqs"]


# ---------------------------------------------------------------------------
# plan
# ---------------------------------------------------------------------------

def test_plan_hand_cases():
    for case in json.load(open(os.path.join(GOLDEN, "plan_cases.json")))["cases"]:
        status, recs = gpu_plan(case["cu"], case["P"])
        assert status == 0
        for r, e in enumerate(case["shards"]):
            a = recs[r]
            got = [a["local_cu"], a["pre_num_ranks"], a["is_first_rank"], a["post_num_ranks"],
                   a["is_last_rank"], a["pre_num_conv_tokens"], a["start_seq_idx"]]
            assert got == e, (case["name"], r)


@pytest.mark.parametrize("trial", range(40))
def test_plan_random(trial):
    r = np.random.default_rng(trial)
    P = int(r.choice([1, 2, 3, 5, 8, 33, 64]))
    part = int(r.integers(1, 50))
    T = P * part
    cuts = np.sort(r.integers(0, T + 1, size=int(r.integers(0, 80))))
    compare_plan(np.concatenate([[0], cuts, [T]]), P)


@pytest.mark.parametrize("name", ["tiny", "packed_varlen", "long", "ragged", "million"])
def test_plan_configs(name):
    w = W.CONFIGS[name]()
    compare_plan(w.cu_seqlens(), w.n_shards)
    for P in (1, 2, 16, 64):
        if w.T % P == 0:
            compare_plan(w.cu_seqlens(), P)


def test_plan_bad_cu_sets_status():
    for cu, P in (([0, 5, 3, 8], 2), ([1, 4, 8], 2), ([0, 4, 9], 2), ([0, 1], 2)):
        status, _ = gpu_plan(cu, P)
        assert status == 6, cu


# ---------------------------------------------------------------------------
# conv
# ---------------------------------------------------------------------------

def conv_case(dtype, Kc, bias, T=300, C=64, seed=0):
    w = W.Workload("conv", T, 1, 1, 32, 32, dtype, 1, seed, (T,), conv_k=Kc, conv_bias=bias)
    x = W.fill(seed, W.TID_X, C, (0, T), (0, C), dtype=w.dt)
    cw = W.fill(seed, W.TID_CONV_W, Kc, (0, C), (0, Kc), b=0.5, dtype=w.dt)
    cb = W.fill(seed, W.TID_CONV_B, C, (0, 1), (0, C), b=0.5, dtype=w.dt)[0] if bias else None
    return x, cw, cb


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("Kc", [1, 2, 3, 4])
@pytest.mark.parametrize("bias", [False, True])
def test_conv_vs_oracle(dtype, Kc, bias):
    import linear_attention_sequence_device_gb300 as g
    x, cw, cb = conv_case(dtype, Kc, bias)
    cu = np.array([0, 1, 3, 64, 64, 150, 300], dtype=np.int32)
    y = g.gdn_conv_silu(to_dev(x, dtype), to_dev(cw, dtype), None if cb is None else to_dev(cb, dtype),
                        torch.from_numpy(cu).to(dev()))
    exp = oracle.conv_silu(W.as_f64(x, dtype), W.as_f64(cw, dtype),
                           None if cb is None else W.as_f64(cb, dtype), cu)
    assert_close(f64(y), exp, dtype, "conv")
    if dtype == "f32":
        assert rel_l2(f64(y), exp) < 1e-6


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_conv_halo(dtype):
    import linear_attention_sequence_device_gb300 as g
    x, cw, _ = conv_case(dtype, 4, False, T=200, C=128, seed=3)
    xd, wd = to_dev(x, dtype), to_dev(cw, dtype)
    full = g.gdn_conv_silu(xd, wd, None, torch.tensor([0, 200], dtype=torch.int32, device=dev()))
    for split, hl in ((64, 3), (70, 3), (101, 2), (33, 1)):
        halo = xd[split - 3:split].contiguous()
        part = g.gdn_conv_silu(xd[split:], wd, None,
                               torch.tensor([0, 200 - split], dtype=torch.int32, device=dev()),
                               halo=halo, halo_len=hl)
        if hl == 3:  # the whole history: bit-identical to the unsharded conv
            assert torch.equal(part, full[split:])
        exp = oracle.conv_silu(W.as_f64(x[split:], dtype), W.as_f64(cw, dtype), None, [0, 200 - split],
                               halo=W.as_f64(x[split - 3:split], dtype), halo_len=hl)
        assert_close(f64(part), exp, dtype, f"conv halo {split}/{hl}")


# ---------------------------------------------------------------------------
# chunked gated delta rule
# ---------------------------------------------------------------------------

CHUNK_CASES = [
    # dtype, Hk, Hv, dk, dv, lengths, h0_std, g_shift
    ("f32", 2, 2, 32, 32, (256,), 0.0, 0.0),
    ("f32", 1, 2, 64, 32, (100, 0, 37, 150), 0.1, -3.0),
    ("f32", 2, 2, 128, 64, (65, 130), 0.05, 0.0),
    ("bf16", 2, 4, 32, 32, (1, 63, 64, 65, 0, 300), 0.05, 0.0),
    ("bf16", 2, 4, 64, 64, (200, 129), 0.0, -4.0),
    ("bf16", 2, 2, 128, 128, (700, 33, 64), 0.02, 0.0),
    ("bf16", 1, 2, 64, 128, (257,), 0.0, 0.0),
    ("bf16", 2, 2, 128, 64, (190,), 0.1, -2.0),
    ("bf16", 1, 1, 128, 32, (128, 5), 0.0, 0.0),
    ("bf16", 2, 2, 32, 128, (99,), 0.0, 0.0),
    # strongly decaying gates (g ~ -softplus(z + 4) ~ -4 per token): the gate
    # range inside a chunk exceeds what split exponentials can hold in fp32
    ("bf16", 2, 2, 128, 128, (300, 77), 0.05, 4.0),
    ("bf16", 1, 2, 128, 128, (190,), 0.0, 1.5),
    # empty sequences on the tensor-core path: their final state is h0
    ("bf16", 2, 2, 128, 128, (0, 130, 0, 70, 0), 0.05, 0.0),
]


def make_chunk_workload(case, seed=11):
    dtype, Hk, Hv, dk, dv, lengths, h0_std, g_shift = case
    return W.Workload("chunk", int(sum(lengths)), Hk, Hv, dk, dv, dtype, 1, seed, tuple(lengths),
                      h0_std=h0_std, g_shift=g_shift)


@pytest.mark.parametrize("case", CHUNK_CASES, ids=lambda c: f"{c[0]}-{c[3]}x{c[4]}-{len(c[5])}seq")
def test_chunk_fwd_vs_oracle(case):
    import linear_attention_sequence_device_gb300 as g
    w = make_chunk_workload(case)
    host, d = chunk_inputs(w)
    g.binding.device_timeouts(reset=True)
    o, hf = g.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu"], h0=d["h0"])
    assert g.binding.device_timeouts() == 0
    o_ref, hf_ref = oracle.gdn_forward(host["q"], host["k"], host["v"], host["g"], host["beta"],
                                       host["h0"], w.cu_seqlens(), w.scale)
    assert_close(f64(o), o_ref, w.dtype, "o")
    assert_close(f64(hf), hf_ref, w.dtype, "h_final")


@pytest.mark.gpu
def test_chunk_fwd_split_sequences_match_unsplit():
    """Sequences of 20, 13 and 3 chunks (bf16, d = 128): with a workspace the
    13-chunk sequence runs as two chained halves (its length lies between half
    and 0.7 of the longest); both orders match the oracle and no wait expires.
    The split falls on a chunk boundary and hands over the fp32 state as is,
    so the two orders agree bit for bit."""
    import linear_attention_sequence_device_gb300 as g
    w = make_chunk_workload(("bf16", 2, 4, 128, 128, (1280, 800, 150), 0.05, 0.5))
    host, d = chunk_inputs(w)
    o_ref, hf_ref = oracle.gdn_forward(host["q"], host["k"], host["v"], host["g"], host["beta"],
                                       host["h0"], w.cu_seqlens(), w.scale)
    g.binding.device_timeouts(reset=True)
    outs = []
    for ws in (None, False):  # per-call workspace (splitting) / none (longest-first only)
        o, hf = g.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu"], h0=d["h0"],
                                workspace=ws)
        assert_close(f64(o), o_ref, w.dtype, "o")
        assert_close(f64(hf), hf_ref, w.dtype, "h_final")
        outs.append((o, hf))
    assert g.binding.device_timeouts() == 0
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])


def test_expired_handover_wait_reports_timeout():
    """A second half whose first half never publishes its final state (the
    gdn_debug_set_handover hook) waits out a 2 ms limit instead of hanging:
    the kernel stops early, writes GDN_ERR_TIMEOUT (7) into the launch's
    status word (word 2 of the gdn_chunk_fwd workspace; the plan's word for
    gdn_shard_fwd) and counts a timeout.  The next launches on the same
    context run normally and match the oracle."""
    import linear_attention_sequence_device_gb300 as g
    b = g.binding
    w = make_chunk_workload(("bf16", 2, 4, 128, 128, (1280, 800, 150), 0.05, 0.5))
    host, d = chunk_inputs(w)
    ws = torch.zeros(b.chunk_fwd_workspace_size(w.N, w.Hv, 128, 128, torch.bfloat16), dtype=torch.uint8,
                     device=dev())
    wp = W.Workload("handover", 2240, 2, 4, 128, 128, "bf16", 1, 13, (1280, 800, 160))
    _, dp = path_inputs(wp)
    b.device_timeouts(reset=True)
    try:
        b.debug_set_handover(2_000_000, publish=False)
        g.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu"], h0=d["h0"], workspace=ws)
        _, _, plan = g.gdn_shard_fwd(dp["x"], dp["conv_w"], None, dp["g"], dp["beta"], dp["cu"], wp.Hk, wp.Hv,
                                     wp.dk, wp.dv, 1, want_plan=True)
        torch.cuda.synchronize()
    finally:
        b.debug_set_handover()
    assert int(ws.view(torch.int32)[2]) == 7
    assert int(plan[0]) == 7
    assert b.device_timeouts(reset=True) >= 2
    o, hf = g.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu"], h0=d["h0"], workspace=ws)
    _, _, plan = g.gdn_shard_fwd(dp["x"], dp["conv_w"], None, dp["g"], dp["beta"], dp["cu"], wp.Hk, wp.Hv,
                                 wp.dk, wp.dv, 1, want_plan=True)
    torch.cuda.synchronize()
    assert int(ws.view(torch.int32)[2]) == 0 and int(plan[0]) == 0
    assert b.device_timeouts() == 0
    o_ref, hf_ref = oracle.gdn_forward(host["q"], host["k"], host["v"], host["g"], host["beta"],
                                       host["h0"], w.cu_seqlens(), w.scale)
    assert_close(f64(o), o_ref, w.dtype, "o")
    assert_close(f64(hf), hf_ref, w.dtype, "h_final")


def test_chunk_fwd_schedule_many_sequences():
    """300 sequences (bf16, d = 128), most short, a few between half and 0.7 of
    the longest: the launch's schedule words, read back, hold every item once
    (whole, or as two halves of the right sizes), longest first within each
    group with every first half ahead of the second halves, and each of the
    persistent CTAs (one per SM) took every ticket it ran plus one past the
    end; the outputs match the oracle."""
    import linear_attention_sequence_device_gb300 as g
    rng = np.random.default_rng(5)
    lengths = [int(x) for x in rng.integers(0, 121, size=295)] + [4000, 2560, 2560, 2560, 2200]
    rng.shuffle(lengths)
    w = make_chunk_workload(("bf16", 1, 2, 128, 128, tuple(lengths), 0.02, 0.0))
    host, d = chunk_inputs(w)
    S, m = len(lengths), 2
    ws = torch.zeros(g.binding.chunk_fwd_workspace_size(S, 2, 128, 128, torch.bfloat16), dtype=torch.uint8,
                     device=dev())
    g.binding.device_timeouts(reset=True)
    o, hf = g.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu"], h0=d["h0"], workspace=ws)
    words = ws.view(torch.int32).cpu().numpy()
    assert g.binding.device_timeouts() == 0
    n = int(words[1])
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert words[0] == n * m + min(sms, 2 * S * m)   # one ticket past the end per CTA
    assert words[2] == 0                              # status word: no wait expired
    off = 4 + S * m + ((4 + S * m) & 1)
    ent = words[off:off + 2 * n].reshape(n, 2)
    items, parts, first = ent[:, 0] & 0xFFFF, ent[:, 0] >> 16, ent[:, 1]
    chunks = [(L + 63) // 64 for L in lengths]
    seen = {}
    for x, pt in zip(items, parts):
        seen.setdefault(int(x), []).append(int(pt))
    assert sorted(seen) == list(range(S))
    split = [x for x, ps in seen.items() if sorted(ps) == [1, 2]]
    assert all(ps == [0] or sorted(ps) == [1, 2] for ps in seen.values())
    assert sorted(chunks[x] for x in split) == [35, 40, 40, 40]
    size = [chunks[x] if pt == 0 else (f if pt == 1 else chunks[x] - f)
            for x, pt, f in zip(items, parts, first)]
    assert all(f == (chunks[x] + 1) // 2 for x, pt, f in zip(items, parts, first) if pt)
    last_first = max(r for r in range(n) if parts[r] == 1)
    assert all(r > last_first for r in range(n) if parts[r] == 2)
    grp = [0 if pt == 1 or (pt == 0 and 2 * chunks[x] > 63) else 1 for x, pt in zip(items, parts)]
    assert grp == sorted(grp)
    for r in range(n - 1):
        if grp[r] == grp[r + 1]:
            assert size[r] >= size[r + 1]
    o_ref, hf_ref = oracle.gdn_forward(host["q"], host["k"], host["v"], host["g"], host["beta"],
                                       host["h0"], w.cu_seqlens(), w.scale)
    assert_close(f64(o), o_ref, w.dtype, "o")
    assert_close(f64(hf), hf_ref, w.dtype, "h_final")


def test_chunk_fwd_strided_views_and_l2norm():
    """q/k/v as column slices of one fused [T, C] buffer; q/k L2-normalised in kernel."""
    import linear_attention_sequence_device_gb300 as g
    T, Hk, Hv, dk, dv = 333, 2, 4, 64, 32
    C = 2 * Hk * dk + Hv * dv
    x = W.fill(5, W.TID_X, C, (0, T), (0, C), dtype=W.DT_BF16)
    xd = to_dev(x, "bf16")
    q = xd[:, :Hk * dk].view(T, Hk, dk)
    k = xd[:, Hk * dk:2 * Hk * dk].view(T, Hk, dk)
    v = xd[:, 2 * Hk * dk:].view(T, Hv, dv)
    gg = W.fill(5, W.TID_G, Hv, (0, T), (0, Hv), kind=W.KIND_NEG_SOFTPLUS, dtype=W.DT_F32)
    bb = W.fill(5, W.TID_BETA, Hv, (0, T), (0, Hv), kind=W.KIND_SIGMOID, dtype=W.DT_BF16)
    cu = np.array([0, 100, 333], dtype=np.int32)
    o, hf = g.gdn_chunk_fwd(q, k, v, to_dev(gg, "f32"), to_dev(bb, "bf16"),
                            torch.from_numpy(cu).to(dev()), l2norm=True)
    xf = W.as_f64(x, "bf16")
    o_ref, hf_ref = oracle.gdn_forward(xf[:, :Hk * dk].reshape(T, Hk, dk),
                                       xf[:, Hk * dk:2 * Hk * dk].reshape(T, Hk, dk),
                                       xf[:, 2 * Hk * dk:].reshape(T, Hv, dv), gg.astype(np.float64),
                                       W.as_f64(bb, "bf16"), None, cu, dk ** -0.5, l2norm=True)
    assert_close(f64(o), o_ref, "bf16", "o")
    assert_close(f64(hf), hf_ref, "bf16", "h_final")


def test_chunk_fwd_resume_equals_one_call():
    import linear_attention_sequence_device_gb300 as g
    w = make_chunk_workload(("bf16", 2, 2, 128, 128, (640,), 0.0, -3.0))
    _, d = chunk_inputs(w)
    o, hf = g.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu"])
    cut = 192
    cu1 = torch.tensor([0, cut], dtype=torch.int32, device=dev())
    cu2 = torch.tensor([0, 640 - cut], dtype=torch.int32, device=dev())
    o1, h1 = g.gdn_chunk_fwd(d["q"][:cut], d["k"][:cut], d["v"][:cut], d["g"][:cut],
                             d["beta"][:cut], cu1)
    o2, h2 = g.gdn_chunk_fwd(d["q"][cut:], d["k"][cut:], d["v"][cut:], d["g"][cut:],
                             d["beta"][cut:], cu2, h0=h1)
    assert rel_l2(f64(torch.cat([o1, o2])), f64(o)) < 1e-2
    assert rel_l2(f64(h2), f64(hf)) < 1e-2


@pytest.mark.parametrize("case", [CHUNK_CASES[0], CHUNK_CASES[2], CHUNK_CASES[5], CHUNK_CASES[7],
                                  CHUNK_CASES[3]], ids=lambda c: f"{c[0]}-{c[3]}x{c[4]}")
def test_chunk_summary_vs_oracle(case):
    import linear_attention_sequence_device_gb300 as g
    w = make_chunk_workload(case[:6] + (0.0, -3.0))
    host, d = chunk_inputs(w)
    M, N = g.gdn_chunk_summary(d["k"], d["v"], d["g"], d["beta"], d["cu"])
    M_ref, N_ref = oracle.gdn_summary(host["k"], host["v"], host["g"], host["beta"], w.cu_seqlens())
    assert_close(f64(M), M_ref, w.dtype, "M")
    assert_close(f64(N), N_ref, w.dtype, "N")


@pytest.mark.parametrize("dk,dv,P,Hv", [(32, 32, 2, 3), (64, 128, 5, 3), (128, 128, 64, 3), (128, 64, 7, 3),
                                         (128, 128, 9, 40), (64, 64, 4, 80)])
def test_state_combine_vs_oracle(dk, dv, P, Hv):
    """16-column state tiles while the CTAs fit the SMs (few heads), else 32."""
    import linear_attention_sequence_device_gb300 as g
    r = np.random.default_rng(dk + dv + P)
    M = r.standard_normal((P, Hv, dk, dk)) / np.sqrt(dk) * 0.9
    N = r.standard_normal((P, Hv, dk, dv))
    S0 = r.standard_normal((Hv, dk, dv))
    for s0 in (None, S0):
        got = g.gdn_state_combine(torch.tensor(M, dtype=torch.float32, device=dev()),
                                  torch.tensor(N, dtype=torch.float32, device=dev()),
                                  None if s0 is None else torch.tensor(s0, dtype=torch.float32, device=dev()))
        exp = oracle.state_combine(M.astype(np.float32).astype(np.float64),
                                   N.astype(np.float32).astype(np.float64),
                                   None if s0 is None else s0.astype(np.float32).astype(np.float64))
        assert rel_l2(f64(got), exp) < 1e-5


def test_zz_no_device_wait_expired():
    """No bounded tensor-core wait expired during the kernel tests above."""
    import linear_attention_sequence_device_gb300 as g
    torch.cuda.synchronize()
    assert g.binding.device_timeouts() == 0


# ---------------------------------------------------------------------------
# head-major layout (the Ulysses wrapper's per-rank view, on one device)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_relayout_round_trip_is_exact(dtype):
    """[T, H, d] token-strided -> dense [H, T, d] -> back: bit-exact, and the
    head-major tensor is the plain transpose."""
    import linear_attention_sequence_device_gb300 as g
    T, H, d, extra = 333, 5, 64, 24
    x = W.fill(9, W.TID_X, H * d + extra, (0, T), (0, H * d + extra), dtype=W.DT_BF16 if dtype == "bf16" else W.DT_F32)
    xd = to_dev(x, dtype)
    xv = xd[:, :H * d].view(T, H, d)
    y = g.binding.to_head_major(xv)
    assert torch.equal(y, xv.permute(1, 0, 2).contiguous())
    back = torch.zeros_like(xd)
    g.binding.to_token_major(y, out=back[:, :H * d].view(T, H, d))
    assert torch.equal(back[:, :H * d], xd[:, :H * d])
    assert bool((back[:, H * d:] == 0).all())


@pytest.mark.parametrize("case", [CHUNK_CASES[5], CHUNK_CASES[4], CHUNK_CASES[1], CHUNK_CASES[12]],
                         ids=lambda c: f"{c[0]}-{c[3]}x{c[4]}")
def test_chunk_fwd_heads_matches_token_major(case):
    """The head-major chunked forward on transposed inputs gives the
    token-major call's outputs bit for bit (same arithmetic), and both match
    the oracle."""
    import linear_attention_sequence_device_gb300 as g
    w = make_chunk_workload(case)
    host, d = chunk_inputs(w)
    o_t, hf_t = g.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu"], h0=d["h0"])
    qh, kh, vh = (g.binding.to_head_major(d[n]) for n in ("q", "k", "v"))
    o_h, hf_h = g.binding.gdn_chunk_fwd_heads(qh, kh, vh, d["g"], d["beta"], d["cu"], h0=d["h0"])
    o_back = g.binding.to_token_major(o_h)
    assert torch.equal(o_back, o_t) and torch.equal(hf_h, hf_t)
    o_ref, hf_ref = oracle.gdn_forward(host["q"], host["k"], host["v"], host["g"], host["beta"],
                                       host["h0"], w.cu_seqlens(), w.scale)
    assert_close(f64(o_back), o_ref, w.dtype, "o")
    assert_close(f64(hf_h), hf_ref, w.dtype, "h_final")
