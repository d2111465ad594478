"""C-ABI checks that need no GPU: the library loads, exports every function
that include/gdn_cp.h declares, and rejects bad arguments on the host with
the documented status codes before touching the device."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gdn_cp.h")


@pytest.fixture(scope="module")
def lib():
    from linear_attention_sequence_device_gb300 import build, binding
    build.build_library()
    return binding.load()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\*?\s*(gdn_[a-z_0-9]+)\s*\(",
                                 src, flags=re.M)))


def test_every_declared_symbol_is_exported(lib):
    from linear_attention_sequence_device_gb300 import binding
    names = declared_functions()
    assert len(names) >= 10, names
    for n in names:
        assert hasattr(lib, n), n
        assert n in binding.SIGNATURES, n


def test_status_strings(lib):
    for code, name in [(0, b"GDN_OK"), (4, b"GDN_ERR_NOT_DIVISIBLE"), (9, b"GDN_ERR_WORKSPACE")]:
        assert lib.gdn_status_string(code) == name


def test_plan_words(lib):
    assert lib.gdn_cp_plan_words(3, 2) == 1 + 2 * 9 + 2 * 2 * 4  # records, local cu, local sequence map
    assert lib.gdn_cp_plan_words(0, 2) == 0


FAKE = ctypes.c_void_p(4096)  # never dereferenced: every call below fails on the host


def shard_call(lib, **kw):
    a = dict(x=FAKE, w=FAKE, b=None, conv_k=4, g=FAKE, beta=FAKE, h0=None, cu=FAKE, N=1, T=256,
             Hk=2, Hv=2, dk=32, dv=32, scale=0.1, flags=1, P=2, dt=0, ws=FAKE, ws_bytes=1 << 40,
             o=FAKE, hf=None, plan=None)
    a.update(kw)
    st = lib.gdn_shard_fwd(a["x"], a["w"], a["b"], a["conv_k"], a["g"], a["beta"], a["h0"],
                           a["cu"], a["N"], a["T"], a["Hk"], a["Hv"], a["dk"], a["dv"], a["scale"],
                           a["flags"], a["P"], a["dt"], a["ws"], a["ws_bytes"], a["o"], a["hf"],
                           a["plan"], None)
    return st, lib.gdn_last_error().decode()


def test_shard_fwd_host_errors(lib):
    assert shard_call(lib, T=250, P=8)[0] == 4                       # not divisible
    assert shard_call(lib, T=16, P=8)[0] == 5                        # shard 2 < halo 3
    assert shard_call(lib, dk=48)[0] == 2                            # unsupported dk
    assert shard_call(lib, Hk=3, Hv=4)[0] == 2                       # Hv % Hk
    assert shard_call(lib, dt=7)[0] == 3                             # dtype
    assert shard_call(lib, conv_k=5)[0] == 2
    assert shard_call(lib, x=None)[0] == 1
    st, msg = shard_call(lib, ws_bytes=16)
    assert st == 9 and "workspace" in msg
    assert shard_call(lib, T=4, P=8)[0] == 1                         # fewer tokens than shards


def test_chunk_fwd_host_errors(lib):
    def call(**kw):
        a = dict(q=FAKE, k=FAKE, v=FAKE, ldq=64, ldk=64, ldv=64, dt=1, T=10, Hk=2, Hv=2, dk=32,
                 dv=32, N=1)
        a.update(kw)
        return lib.gdn_chunk_fwd(a["q"], a["k"], a["v"], a["ldq"], a["ldk"], a["ldv"], a["dt"],
                                 FAKE, FAKE, None, FAKE, a["N"], a["T"], a["Hk"], a["Hv"], a["dk"],
                                 a["dv"], 0.1, 0, FAKE, None, None, 0, None)
    assert call(ldq=60) == 1          # stride below Hk * dk
    assert call(ldq=68) == 1          # stride not a multiple of 8
    assert call(q=ctypes.c_void_p(4104)) == 1  # misaligned
    assert call(N=0) == 1
    assert call(dv=96) == 2


def test_chunk_fwd_workspace_contract(lib):
    """The optional work-queue workspace: its size is a multiple of 256 bytes
    that grows with the sequence count (0 for invalid arguments); a smaller or
    misaligned workspace is rejected on the host before any launch."""
    size = lambda n, hv=4, d=128, dt=1: lib.gdn_chunk_fwd_workspace_size(n, hv, d, d, dt)
    assert size(0) == 0 and size(3, hv=0) == 0
    for n in (1, 7, 300):
        assert size(n) > 0 and size(n) % 256 == 0
    assert size(1) <= size(7) <= size(300)
    assert size(300, hv=8) >= size(300, hv=4)

    def call(ws, ws_bytes):
        return lib.gdn_chunk_fwd(FAKE, FAKE, FAKE, 512, 512, 512, 1, FAKE, FAKE, None, FAKE, 3, 256, 4, 4,
                                 128, 128, 0.1, 0, FAKE, FAKE, ws, ws_bytes, None)
    need = size(3)
    assert call(FAKE, need - 1) == 9
    assert "workspace" in lib.gdn_last_error().decode()
    assert call(ctypes.c_void_p(4100), need) == 9  # not 16-byte aligned


def test_conv_host_errors(lib):
    def call(**kw):
        a = dict(C=64, K=4, halo=None, hl=0, T=8)
        a.update(kw)
        return lib.gdn_conv_silu(FAKE, a["C"], 1, a["T"], a["C"], FAKE, None, a["K"], FAKE, 1,
                                 a["halo"], a["hl"], FAKE, a["C"], None)
    assert call(C=60) == 2
    assert call(K=0) == 2
    assert call(hl=3) == 1            # halo_len > 0 without a halo pointer
    assert call(hl=4, halo=FAKE) == 1  # halo_len > conv_k - 1


def test_backward_host_errors(lib):
    """gdn_chunk_bwd and gdn_shard_bwd reject bad arguments on the host (before
    any launch) with the documented status codes; their workspace queries
    return 0 for unsupported shapes."""
    assert lib.gdn_chunk_bwd_workspace_size(64, 1, 1, 1, 48, 64) == 0
    assert lib.gdn_chunk_bwd_workspace_size(64, 0, 1, 1, 32, 32) == 0
    assert lib.gdn_shard_bwd_workspace_size(64, 1, 2, 1, 1, 32, 96) == 0
    need = lib.gdn_chunk_bwd_workspace_size(64, 1, 2, 2, 32, 32)
    assert need > 0 and need % 256 == 0

    def chunk(**kw):
        a = dict(q=FAKE, ldq=64, dt=1, T=64, N=1, Hk=2, Hv=2, dk=32, dv=32, flags=0, cu=FAKE, dh0=FAKE,
                 ws=FAKE, ws_bytes=need)
        a.update(kw)
        return lib.gdn_chunk_bwd(a["q"], FAKE, FAKE, a["ldq"], 64, 64, a["dt"], FAKE, FAKE, None, FAKE, None,
                                 a["cu"], a["N"], a["T"], a["Hk"], a["Hv"], a["dk"], a["dv"], 0.1, a["flags"],
                                 FAKE, FAKE, FAKE, FAKE, FAKE, a["dh0"], a["ws"], a["ws_bytes"], None)
    assert chunk(dk=48) == 2                        # unsupported head size
    assert chunk(dt=7) == 3                         # dtype
    assert chunk(N=0) == 1
    assert chunk(cu=None) == 1 and chunk(dh0=None) == 1
    assert chunk(flags=4) == 1                      # unknown flag bit
    assert chunk(ws_bytes=need - 1) == 9            # workspace too small
    assert chunk(ws=ctypes.c_void_p(4096 + 16)) == 9  # workspace not 256-byte aligned
    assert chunk(ldq=60) == 1                       # q row stride below Hk * dk
    assert chunk(q=ctypes.c_void_p(4104)) == 1      # q misaligned

    sneed = lib.gdn_shard_bwd_workspace_size(64, 1, 2, 2, 2, 32, 32)
    assert sneed > 0

    def shard(**kw):
        a = dict(T=64, P=2, ws=FAKE, ws_bytes=sneed, flags=0)
        a.update(kw)
        return lib.gdn_shard_bwd(FAKE, FAKE, FAKE, 64, 64, 64, 1, FAKE, FAKE, None, FAKE, None, FAKE, 1, a["T"],
                                 2, 2, 32, 32, 0.1, a["flags"], a["P"], FAKE, FAKE, FAKE, FAKE, FAKE, FAKE,
                                 a["ws"], a["ws_bytes"], None, None)
    assert shard(T=63) == 4                         # not a multiple of n_shards
    assert shard(P=0) == 1
    assert shard(flags=4) == 1
    assert shard(ws_bytes=sneed - 1) == 9


def test_shard_fwd_workspace_sizes(lib):
    """The full workspace adds room for the stored summary operands (bf16,
    d = 128, P > 1: W rows, K~ tiles and e^{G_last} of every shard chunk),
    plus, when the M chains are cut into G segments (2 <= G <= 8, chosen from
    the device's SM count), G fp32 products of 64 KiB per (shard, head);
    otherwise it equals the minimum.  0 for invalid arguments."""
    full = lambda *a: lib.gdn_shard_fwd_workspace_size(*a)
    small = lambda *a: lib.gdn_shard_fwd_workspace_min_size(*a)
    a = (131072, 1, 8, 16, 16, 128, 128, 1)            # bf16, d = 128, P = 8
    extra = full(*a) - small(*a)
    chunks = 8 * 16 * ((131072 // 8 + 63) // 64)
    ops = chunks * (2 * 64 * 128 * 2 + 4)
    assert ops <= extra < ops + 3 * 256 + 8 * 8 * 16 * 65536
    seg = (extra - ops) // (8 * 16 * 65536)            # segments' products (alignment rounds up < 1 KiB)
    assert seg == 0 or 2 <= seg <= 8
    assert extra - ops - seg * 8 * 16 * 65536 < 4 * 256
    for b in ((131072, 1, 1, 16, 16, 128, 128, 1),     # one shard
              (4096, 2, 4, 2, 2, 64, 64, 1),           # other head size
              (4096, 2, 4, 2, 2, 128, 128, 0)):        # fp32
        assert full(*b) == small(*b) > 0
    assert full(0, 0, 1, 1, 1, 128, 128, 1) == 0 and small(0, 0, 1, 1, 1, 128, 128, 1) == 0


def test_internal_shard_count_in_the_workspace(lib):
    """The shard count a gdn_shard_fwd call runs on shows in its workspace:
    plan, conv output, carries (N, S_in, M) and pass-1 schedule are sized for
    it.  One 131072-token sequence with 16 heads on 8 shards (bf16, d = 128)
    runs on 16 internal shards (few chains for the SMs: 148 assumed without
    a GPU); two sequences, fp32 and the million shape keep the caller's
    count."""
    a256 = lambda x: (x + 255) // 256 * 256

    def min_size(T, N, P, Hk, Hv, d, bf16):
        e = 2 if bf16 else 4
        cch = 2 * Hk * d + Hv * d
        carry = P * Hv * d
        tile = 128 if bf16 and d == 128 else (32 if not bf16 else min(d, 64))
        S, m = N + P, Hv * (2 * d // tile)
        o = 4 + S * m
        o += o & 1
        return (a256(4 * lib.gdn_cp_plan_words(N, P)) + a256(T * cch * e) + 2 * a256(carry * d * 4)
                + a256(carry * d * 4) + a256(4 * (o + 4 * S)))

    small = lambda *a: lib.gdn_shard_fwd_workspace_min_size(*a)
    assert small(131072, 1, 8, 16, 16, 128, 128, 1) == min_size(131072, 1, 16, 16, 16, 128, True)
    assert small(131072, 2, 8, 16, 16, 128, 128, 1) == min_size(131072, 2, 8, 16, 16, 128, True)
    assert small(131072, 1, 8, 16, 16, 128, 128, 0) == min_size(131072, 1, 8, 16, 16, 128, False)
    assert small(1048576, 1, 64, 32, 32, 128, 128, 1) == min_size(1048576, 1, 64, 32, 32, 128, True)


def test_m_chain_segments_in_the_workspace(lib):
    """The M chains' segment count shows in the full workspace (G products of
    64 KiB per (shard, head) when G > 1).  Two sequences on 4 shards of 64
    chunks with 16 heads: 32 chains for 296 resident slots (148 SMs assumed
    without a GPU) are cut into 4 segments of 16 chunks; one long sequence
    (16 internal shards, 224 chains of 128 chunks) keeps whole chains, since
    the merge would cost more than the cut saves."""
    a256 = lambda x: (x + 255) // 256 * 256

    def extra(T, N, P, Hv, P_run):
        full = lib.gdn_shard_fwd_workspace_size(T, N, P, 16, Hv, 128, 128, 1)
        small = lib.gdn_shard_fwd_workspace_min_size(T, N, P, 16, Hv, 128, 128, 1)
        chunks = P_run * Hv * ((T // P_run + 63) // 64)
        ops = 2 * a256(chunks * 64 * 128 * 2) + a256(chunks * 4)
        return full - small - ops

    assert extra(16384, 2, 4, 16, 4) == a256(4 * 4 * 16 * 65536)
    assert extra(131072, 1, 8, 16, 16) == 0  # runs on 16 shards of 128 chunks


def test_testing_hooks_are_host_settings(lib):
    """The testing hooks only set host-side launch settings (no device call):
    the split switch takes any int, the hand-over bound rejects a negative
    limit; the defaults are restored."""
    assert lib.gdn_debug_set_split(0) == 0
    assert lib.gdn_debug_set_split(1) == 0
    assert lib.gdn_debug_set_handover(-1, 1) == 1          # GDN_ERR_INVALID_ARG
    assert lib.gdn_debug_set_handover(1_000_000_000, 1) == 0
