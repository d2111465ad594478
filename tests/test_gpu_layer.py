"""GPU parity of gdn_layer_fwd: the wrappers' forward between the projections
(gates from the raw a / b projections, the path on P virtual shards, the
gated RMS norm with z) against the fp64 oracle's layer_forward.

bf16 with d = 128 runs the norm as the tensor-core chunk kernel's output
epilogue and the gates inside its loads; the other shapes run the gates in
their own chunk kernels and the norm as a separate pass.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from tests.parity import assert_close, dev, f64, path_inputs, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    from linear_attention_sequence_device_gb300 import build
    build.build_library()
    import linear_attention_sequence_device_gb300 as g
    g.load()
    return g


def layer_inputs(w):
    host, d = path_inputs(w)
    raw = dict(a=w.a_proj(), b=w.b_proj(), z=w.z(), norm_w=w.norm_w())
    host.update({k: W.as_f64(v, w.dtype) for k, v in raw.items()})
    host.update(A_log=w.A_log().astype(np.float64), dt_bias=w.dt_bias().astype(np.float64))
    d.update({k: to_dev(v, w.dtype) for k, v in raw.items()})
    d.update(A_log=to_dev(w.A_log(), "f32"), dt_bias=to_dev(w.dt_bias(), "f32"))
    return host, d


def run_layer(w, d, P, with_norm=True):
    import linear_attention_sequence_device_gb300 as g
    z = d["z"].view(w.T, w.Hv, w.dv) if with_norm else None
    return g.gdn_layer_fwd(d["x"], d["conv_w"], d["conv_b"], d["a"], d["b"], d["A_log"], d["dt_bias"], z,
                           d["norm_w"] if with_norm else None, d["cu"], w.Hk, w.Hv, w.dk, w.dv, P, h0=d["h0"],
                           want_plan=True)


def oracle_layer(w, host, with_norm=True):
    if not with_norm:
        g, beta = oracle.gates(host["a"], host["b"], host["A_log"], host["dt_bias"])
        return oracle.path_forward(W.as_f64(host["x"], w.dtype), host["conv_w"], host["conv_b"], g, beta,
                                   host["h0"], w.cu_seqlens(), w.Hk, w.Hv, w.dk, w.dv, w.scale)
    return oracle.layer_forward(W.as_f64(host["x"], w.dtype), host["conv_w"], host["conv_b"], host["a"],
                                host["b"], host["A_log"], host["dt_bias"],
                                host["z"].reshape(w.T, w.Hv, w.dv), host["norm_w"], host["h0"],
                                w.cu_seqlens(), w.Hk, w.Hv, w.dk, w.dv, w.scale)


CASES = [
    ("tiny_f32", lambda: W.tiny(), 2),
    ("tiny_f32_P8", lambda: W.tiny(n_shards=8), 8),
    ("packed_bf16_128", lambda: W.Workload("packed_small", 2048, 16, 32, 128, 128, "bf16", 1, 1,
                                           W.lengths_uniform(1, 2048, 64, 700)), 1),
    ("long_bf16_128_P8", lambda: W.long_seq(T=2048, h0_std=0.02), 8),
    # one sequence on 2 shards: the call runs on 4 internal shards
    ("long_bf16_128_P2_internal", lambda: W.long_seq(T=4096, h0_std=0.02), 2),
    # 8 x 32 jobs a pass: the work queue splits every item, M halves included
    ("million_bf16_128_P8_split", lambda: W.million(T=8000, n_shards=8), 8),
    ("ragged_bf16_128_P4", lambda: W.Workload("ragged_small", 2048, 4, 8, 128, 128, "bf16", 4, 3,
                                              W.lengths_geometric(3, 2048, 1.0 / 300.0, 1, 4096)), 4),
    ("bf16_64", lambda: W.Workload("small64", 700, 2, 4, 64, 64, "bf16", 1, 7, (300, 1, 399)), 1),
]


@pytest.mark.parametrize("name,make,P", CASES, ids=[c[0] for c in CASES])
def test_layer_fwd_vs_oracle(name, make, P):
    """End to end against the oracle's layer: y within the relative-L2 bar
    (the max-abs bar is defined for the GDN output on L2-normalised q/k; y is
    normalised per row to unit RMS and gated by silu(z), so it is O(1)-O(10)
    and its bf16 rounding alone can exceed 2e-2), h_final within both bars;
    and the norm itself, element by element, against the oracle's gated norm
    of the GPU's own output o (same call without z): |dy| <= 2^-7 |y| + 1e-5
    for bf16 (output rounding 2^-9, the bf16 o the norm reads, fp32 sums),
    1e-5 |y| + 1e-7 for fp32."""
    w = make()
    host, d = layer_inputs(w)
    y, hf, plan = run_layer(w, d, P)
    y_ref, hf_ref = oracle_layer(w, host)
    assert int(plan[0]) == 0
    assert_close(f64(y), y_ref, w.dtype, f"{name} y", max_abs=False)
    assert_close(f64(hf), hf_ref, w.dtype, f"{name} h_final")
    o, _, _ = run_layer(w, d, P, with_norm=False)
    y_of_o = oracle.gated_rmsnorm(f64(o), host["z"].reshape(w.T, w.Hv, w.dv), host["norm_w"])
    rel, ab = (2.0 ** -7, 1e-5) if w.dtype == "bf16" else (1e-5, 1e-7)
    err = np.abs(f64(y) - y_of_o)
    bad = err > rel * np.abs(y_of_o) + ab
    assert not bad.any(), (f"{name}: {int(bad.sum())} elements off the gated norm of o; worst "
                           f"{float((err - rel * np.abs(y_of_o)).max()):.3e}")


def test_layer_fwd_without_norm_equals_shard_fwd_on_the_gates():
    """z = NULL: y is the path's output on the gates the layer computes; the
    same as gdn_shard_fwd given the oracle's g and beta (rounded as the
    kernel rounds beta) within the bars."""
    import linear_attention_sequence_device_gb300 as g
    w = W.long_seq(T=2048)
    host, d = layer_inputs(w)
    y, hf, _ = run_layer(w, d, 8, with_norm=False)
    y_ref, hf_ref = oracle_layer(w, host, with_norm=False)
    assert_close(f64(y), y_ref, w.dtype, "y")
    assert_close(f64(hf), hf_ref, w.dtype, "h_final")
    gg, bb = oracle.gates(host["a"], host["b"], host["A_log"], host["dt_bias"])
    o, hf2, _ = g.gdn_shard_fwd(d["x"], d["conv_w"], None, torch.tensor(gg, dtype=torch.float32, device=dev()),
                                torch.tensor(bb, dtype=torch.float32, device=dev()).to(torch.bfloat16), d["cu"],
                                w.Hk, w.Hv, w.dk, w.dv, 8)
    assert_close(f64(y), f64(o), w.dtype, "layer vs shard_fwd")
