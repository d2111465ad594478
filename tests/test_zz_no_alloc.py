"""gdn_shard_fwd_noalloc: the sharded forward for callers that cannot
allocate device memory (a plugin handed only its input/output buffers, a
loop that may not call cudaMalloc).  It must give the same results as
gdn_shard_fwd with a caller workspace, call after call, although every call
reuses the library's one fixed scratch array.  Collected last on purpose.
"""
import numpy as np
import pytest
import torch

import workloads as W
from tests.parity import TOL_REL_L2, f64, path_inputs, rel_l2

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def g():
    from linear_attention_sequence_device_gb300 import build
    build.build_library()
    import linear_attention_sequence_device_gb300.binding as b
    b.load()
    return b


def _case(seed, n_shards, T=1024):
    lengths = W.lengths_uniform(seed, T, 100, 700)
    return W.Workload("noalloc", T, 16, 16, 128, 128, "bf16", n_shards, seed, lengths,
                      h0_std=0.02)


def _both(g, w):
    _, d = path_inputs(w)
    args = (d["x"], d["conv_w"], d["conv_b"], d["g"], d["beta"], d["cu"], w.Hk, w.Hv, w.dk, w.dv,
            w.n_shards)
    o_ref, hf_ref, _ = g.gdn_shard_fwd(*args, h0=d["h0"])
    o, hf = g.gdn_shard_fwd_noalloc(*args, h0=d["h0"])
    torch.cuda.synchronize()
    return o, hf, o_ref, hf_ref


def test_noalloc_matches_workspace_path_two_calls(g):
    for w in (_case(21, 4), _case(22, 2), W.tiny()):
        assert g.shard_fwd_workspace_min_size(w.T, w.N, w.n_shards, w.Hk, w.Hv, w.dk, w.dv,
                                              torch.bfloat16 if w.dtype == "bf16" else torch.float32) \
            <= g.NOALLOC_SCRATCH_BYTES
        o, hf, o_ref, hf_ref = _both(g, w)
        assert rel_l2(f64(o), f64(o_ref)) <= TOL_REL_L2[w.dtype], w.name
        assert rel_l2(f64(hf), f64(hf_ref)) <= TOL_REL_L2[w.dtype], w.name


def test_noalloc_split_item_after_a_sharded_call(g):
    """One shard whose sequence lengths make the tensor-core kernel split an
    item into two halves chained through flags in the scratch array, right
    after a multi-shard call has left its own contents there: the flags are
    rewritten by the call, so the result matches gdn_shard_fwd with a fresh
    workspace, and no bounded device wait expires."""
    g.device_timeouts(reset=True)
    _both(g, _case(23, 4))
    w = W.Workload("noalloc_split", 2240, 2, 4, 128, 128, "bf16", 1, 24, (1280, 800, 160), h0_std=0.02)
    o, hf, o_ref, hf_ref = _both(g, w)
    assert rel_l2(f64(o), f64(o_ref)) <= TOL_REL_L2[w.dtype]
    assert rel_l2(f64(hf), f64(hf_ref)) <= TOL_REL_L2[w.dtype]
    assert g.device_timeouts() == 0


def test_noalloc_rejects_problems_beyond_its_scratch(g):
    w = W.long_seq(T=8192)
    _, d = path_inputs(w)
    with pytest.raises(g.GdnError) as e:
        g.gdn_shard_fwd_noalloc(d["x"], d["conv_w"], None, d["g"], d["beta"], d["cu"], w.Hk, w.Hv,
                                w.dk, w.dv, w.n_shards)
    assert e.value.status == 9 and "scratch" in str(e.value)
