// C ABI of libgdncp: host-side validation, status codes and stream-ordered
// launches.  Nothing here allocates memory or synchronises the host.
#include <cstdarg>
#include <cstdio>
#include <cstring>

#include "gdn_internal.cuh"

namespace gdn {

static thread_local char g_err[512] = "";

// Profiling hook: events recorded between the phases of gdn_shard_fwd.
static thread_local cudaEvent_t g_phase_events[8];
static thread_local int g_phase_n = 0;

gdn_status fail(gdn_status s, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof(g_err), fmt, ap);
    va_end(ap);
    return s;
}

gdn_status check_launch(const char* what) {
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(GDN_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
    return GDN_OK;
}

// cudaFuncAttributeMaxDynamicSharedMemorySize, set once per (device, kernel).
gdn_status set_smem_attr(const void* func, size_t bytes) {
    constexpr int kMaxDev = 64, kMaxFn = 32;
    static thread_local const void* done[kMaxDev][kMaxFn] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev)
        return check_launch("cudaGetDevice");
    for (int i = 0; i < kMaxFn; ++i) {
        if (done[dev][i] == func) return GDN_OK;
        if (done[dev][i] == nullptr) {
            if (cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes) !=
                cudaSuccess)
                return check_launch("cudaFuncSetAttribute");
            done[dev][i] = func;
            return GDN_OK;
        }
    }
    if (cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes) != cudaSuccess)
        return check_launch("cudaFuncSetAttribute");
    return GDN_OK;
}

int chunk_col_tile(gdn_dtype dt, int dk, int dv) {
    if (chunk_tc_eligible(dt, dk, dv)) return 128;
    if (dt == GDN_F32) return 32;
    int t = dk < dv ? dk : dv;
    return t < 64 ? t : 64;
}

static bool dim_ok(int d) { return d == 32 || d == 64 || d == 128; }
static bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
static size_t esize(gdn_dtype dt) { return dt == GDN_BF16 ? 2 : 4; }
static size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

int device_sm_count() {
    static int sms[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
    if (!sms[dev]) cudaDeviceGetAttribute(&sms[dev], cudaDevAttrMultiProcessorCount, dev);
    return sms[dev] > 0 ? sms[dev] : 148;
}

// Shards a gdn_shard_fwd call runs on.  The result is the same for any shard
// count (the sharded path equals the unsharded one), so one sequence cut into
// fewer shards than the SMs can hold, whose chains then leave SMs idle in both
// passes, is cut finer inside the call: n_shards * 2^j (j <= 3, dividing T,
// shards of 1024 tokens at least), each doubling kept only if it cuts the
// modelled time by a tenth.  Model, in chunk periods: per pass the longer of
// one shard's chain and the spanning shards' work spread over the SMs, two
// passes, plus one merge step per shard.  Only the tensor-core path (bf16,
// d = 128); the plan a caller receives is always that of its own n_shards.
int internal_shards(int T, int num_seqs, int P, int Hv, int dk, int dv, gdn_dtype dtype) {
    if (P < 2 || num_seqs != 1 || T <= 0 || !chunk_tc_eligible(dtype, dk, dv)) return P;
    const double sms = (double)device_sm_count();
    auto cost = [&](long long Q) {
        const double L = (double)(T / Q) / 64.0, spread = (double)(Q - 1) * Hv * L / sms;
        return 2.0 * (L > spread ? L : spread) + (double)Q;
    };
    long long best = P;
    double bc = cost(P);
    for (long long Q = 2ll * P; Q <= 8ll * P && Q <= 65536 && T % Q == 0 && T / Q >= 1024; Q *= 2) {
        const double c = cost(Q);
        if (c < 0.9 * bc) {
            best = Q;
            bc = c;
        }
    }
    return (int)best;
}

// checks shared by gdn_chunk_fwd / gdn_chunk_summary / gdn_shard_fwd
static gdn_status check_heads(gdn_dtype dt, int T, int num_seqs, int Hk, int Hv, int dk, int dv) {
    if (dt != GDN_F32 && dt != GDN_BF16) return fail(GDN_ERR_DTYPE, "unknown dtype %d", (int)dt);
    if (T < 0 || num_seqs < 1) return fail(GDN_ERR_INVALID_ARG, "T=%d num_seqs=%d", T, num_seqs);
    if (Hk < 1 || Hv < 1 || Hv % Hk != 0)
        return fail(GDN_ERR_UNSUPPORTED_SHAPE, "Hv=%d must be a positive multiple of Hk=%d", Hv, Hk);
    if (Hv > 65535) return fail(GDN_ERR_UNSUPPORTED_SHAPE, "Hv=%d too large", Hv);
    if (!dim_ok(dk) || !dim_ok(dv))
        return fail(GDN_ERR_UNSUPPORTED_SHAPE, "dk=%d dv=%d must be in {32,64,128}", dk, dv);
    return GDN_OK;
}

static gdn_status check_row(const void* p, int64_t ld, int64_t minld, const char* name) {
    if (!p) return fail(GDN_ERR_INVALID_ARG, "%s is NULL", name);
    if (!al16(p)) return fail(GDN_ERR_INVALID_ARG, "%s must be 16-byte aligned", name);
    if (ld < minld || ld % 8 != 0)
        return fail(GDN_ERR_INVALID_ARG, "row stride of %s (%lld) must be >= %lld and a multiple of 8",
                    name, (long long)ld, (long long)minld);
    return GDN_OK;
}

static gdn_status launch_chunk(const ChunkParams& p, gdn_dtype dt, int src, dim3 grid, cudaStream_t s) {
    if (grid.x == 0) return GDN_OK;
    if (chunk_tc_eligible(dt, p.dk, p.dv)) return launch_chunk_tc(p, src, grid, s);
    return dt == GDN_BF16 ? launch_chunk_bf16(p, src, grid, s) : launch_chunk_f32(p, src, grid, s);
}

}  // namespace gdn

using namespace gdn;

extern "C" {

const char* gdn_status_string(gdn_status s) {
    switch (s) {
        case GDN_OK: return "GDN_OK";
        case GDN_ERR_INVALID_ARG: return "GDN_ERR_INVALID_ARG";
        case GDN_ERR_UNSUPPORTED_SHAPE: return "GDN_ERR_UNSUPPORTED_SHAPE";
        case GDN_ERR_DTYPE: return "GDN_ERR_DTYPE";
        case GDN_ERR_NOT_DIVISIBLE: return "GDN_ERR_NOT_DIVISIBLE";
        case GDN_ERR_SHARD_TOO_SHORT: return "GDN_ERR_SHARD_TOO_SHORT";
        case GDN_ERR_BAD_CU_SEQLENS: return "GDN_ERR_BAD_CU_SEQLENS";
        case GDN_ERR_TIMEOUT: return "GDN_ERR_TIMEOUT";
        case GDN_ERR_CUDA: return "GDN_ERR_CUDA";
        case GDN_ERR_WORKSPACE: return "GDN_ERR_WORKSPACE";
    }
    return "GDN_ERR_UNKNOWN";
}

const char* gdn_last_error(void) { return g_err; }

gdn_status gdn_debug_set_phase_events(void* const* events, int32_t n) {
    if (n < 0 || n > 8 || (n > 0 && !events)) return fail(GDN_ERR_INVALID_ARG, "n=%d events=%p", n, (const void*)events);
    for (int i = 0; i < n; ++i) g_phase_events[i] = static_cast<cudaEvent_t>(events[i]);
    g_phase_n = n;
    return GDN_OK;
}

gdn_status gdn_device_timeouts(int32_t* count, int reset) {
    if (!count) return fail(GDN_ERR_INVALID_ARG, "count is NULL");
    int v = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_gdn_timeouts, sizeof(int));
    if (e != cudaSuccess) return fail(GDN_ERR_CUDA, "reading the timeout counter: %s", cudaGetErrorString(e));
    *count = v;
    if (reset) {
        const int zero = 0;
        e = cudaMemcpyToSymbol(g_gdn_timeouts, &zero, sizeof(int));
        if (e != cudaSuccess) return fail(GDN_ERR_CUDA, "resetting the timeout counter: %s", cudaGetErrorString(e));
    }
    return GDN_OK;
}

int64_t gdn_cp_plan_words(int32_t num_seqs, int32_t n_shards) {
    if (num_seqs < 1 || n_shards < 1) return 0;
    return 1 + (int64_t)n_shards * GDN_PLAN_NFIELDS + 2 * (int64_t)n_shards * ((int64_t)num_seqs + 1);
}

gdn_status gdn_cp_plan(const int32_t* cu_seqlens, int32_t num_seqs, int32_t n_shards, int32_t* plan,
                       void* stream) {
    if (!cu_seqlens || !plan) return fail(GDN_ERR_INVALID_ARG, "cu_seqlens/plan is NULL");
    if (num_seqs < 1) return fail(GDN_ERR_INVALID_ARG, "num_seqs=%d < 1", num_seqs);
    if (n_shards < 1 || n_shards > 65536)
        return fail(GDN_ERR_INVALID_ARG, "n_shards=%d not in [1, 65536]", n_shards);
    return launch_plan(cu_seqlens, num_seqs, n_shards, plan, (cudaStream_t)stream);
}

gdn_status gdn_conv_silu(const void* x, int64_t ldx, gdn_dtype dtype, int32_t T, int32_t channels,
                         const void* w, const void* bias, int32_t conv_k, const int32_t* cu_seqlens,
                         int32_t num_seqs, const void* halo, int32_t halo_len, void* y, int64_t ldy,
                         void* stream) {
    if (dtype != GDN_F32 && dtype != GDN_BF16) return fail(GDN_ERR_DTYPE, "unknown dtype %d", (int)dtype);
    if (T < 0 || num_seqs < 1 || channels < 1)
        return fail(GDN_ERR_INVALID_ARG, "T=%d num_seqs=%d channels=%d", T, num_seqs, channels);
    if (channels % 8 != 0) return fail(GDN_ERR_UNSUPPORTED_SHAPE, "channels=%d not a multiple of 8", channels);
    if (conv_k < 1 || conv_k > 4) return fail(GDN_ERR_UNSUPPORTED_SHAPE, "conv_k=%d not in 1..4", conv_k);
    if (halo_len < 0 || halo_len > conv_k - 1)
        return fail(GDN_ERR_INVALID_ARG, "halo_len=%d not in [0, conv_k-1]", halo_len);
    if (halo_len > 0 && (!halo || !al16(halo)))
        return fail(GDN_ERR_INVALID_ARG, "halo must be a 16-byte aligned pointer when halo_len > 0");
    if (!w || !cu_seqlens) return fail(GDN_ERR_INVALID_ARG, "w/cu_seqlens is NULL");
    if (T == 0) return GDN_OK;
    gdn_status st;
    if ((st = check_row(x, ldx, channels, "x")) != GDN_OK) return st;
    if ((st = check_row(y, ldy, channels, "y")) != GDN_OK) return st;
    return launch_conv(x, ldx, dtype, T, channels, w, bias, conv_k, cu_seqlens, num_seqs, halo,
                       halo_len, y, ldy, nullptr, 1, (cudaStream_t)stream);
}

gdn_status gdn_chunk_fwd(const void* q, const void* k, const void* v, int64_t ldq, int64_t ldk,
                         int64_t ldv, gdn_dtype dtype, const float* g, const void* beta,
                         const float* h0, const int32_t* cu_seqlens, int32_t num_seqs, int32_t T,
                         int32_t Hk, int32_t Hv, int32_t dk, int32_t dv, float scale, uint32_t flags,
                         void* o, float* h_final, void* workspace, size_t workspace_bytes, void* stream) {
    gdn_status st = check_heads(dtype, T, num_seqs, Hk, Hv, dk, dv);
    if (st != GDN_OK) return st;
    if (!cu_seqlens) return fail(GDN_ERR_INVALID_ARG, "cu_seqlens is NULL");
    const size_t need = gdn_chunk_fwd_workspace_size(num_seqs, Hv, dk, dv, dtype);
    if (workspace && workspace_bytes < need)
        return fail(GDN_ERR_WORKSPACE, "workspace of %zu bytes < required %zu", workspace_bytes, need);
    if (workspace && !al16(workspace)) return fail(GDN_ERR_WORKSPACE, "workspace must be 16-byte aligned");
    if (T > 0) {
        if ((st = check_row(q, ldq, (int64_t)Hk * dk, "q")) != GDN_OK) return st;
        if ((st = check_row(k, ldk, (int64_t)Hk * dk, "k")) != GDN_OK) return st;
        if ((st = check_row(v, ldv, (int64_t)Hv * dv, "v")) != GDN_OK) return st;
        if (!g || !beta || !o) return fail(GDN_ERR_INVALID_ARG, "g/beta/o is NULL");
        if (!al16(o)) return fail(GDN_ERR_INVALID_ARG, "o must be 16-byte aligned");
    }
    if (h_final && (reinterpret_cast<uintptr_t>(h_final) & 7u))
        return fail(GDN_ERR_INVALID_ARG, "h_final must be 8-byte aligned");
    ChunkParams p{};
    p.q = q; p.k = k; p.v = v; p.ldq = ldq; p.ldk = ldk; p.ldv = ldv;
    p.g = g; p.beta = beta; p.h0 = h0; p.cu = cu_seqlens;
    p.num_seqs = num_seqs; p.T = T; p.Hk = Hk; p.Hv = Hv; p.dk = dk; p.dv = dv;
    p.scale = scale; p.flags = flags; p.o = o; p.h_final = h_final;
    p.col_tile = chunk_col_tile(dtype, dk, dv);
    set_token_major(p);
    if (workspace && T > 0 && chunk_tc_eligible(dtype, dk, dv))
        p.sched = static_cast<int32_t*>(workspace);  // work queue, filled by the order kernel before the chunk kernel
    dim3 grid(num_seqs, Hv, dv / p.col_tile);
    return launch_chunk(p, dtype, JOBS_SEQS, grid, (cudaStream_t)stream);
}

size_t gdn_chunk_bwd_workspace_size(int32_t T, int32_t num_seqs, int32_t Hk, int32_t Hv, int32_t dk, int32_t dv) {
    if (T < 0 || num_seqs < 1 || Hk < 1 || Hv < 1 || !dim_ok(dk) || !dim_ok(dv)) return 0;
    return chunk_bwd_workspace_bytes(T, num_seqs, Hk, Hv, dk, dv);
}

gdn_status gdn_chunk_bwd(const void* q, const void* k, const void* v, int64_t ldq, int64_t ldk, int64_t ldv,
                         gdn_dtype dtype, const float* g, const void* beta, const float* h0, const void* dout,
                         const float* dh_final, const int32_t* cu_seqlens, int32_t num_seqs, int32_t T, int32_t Hk,
                         int32_t Hv, int32_t dk, int32_t dv, float scale, uint32_t flags, float* dq, float* dk_,
                         float* dv_, float* dg, float* dbeta, float* dh0, void* workspace, size_t workspace_bytes,
                         void* stream) {
    gdn_status st = check_heads(dtype, T, num_seqs, Hk, Hv, dk, dv);
    if (st != GDN_OK) return st;
    if (!cu_seqlens || !dh0) return fail(GDN_ERR_INVALID_ARG, "cu_seqlens/dh0 is NULL");
    if (flags & ~(uint32_t)GDN_QK_L2NORM) return fail(GDN_ERR_INVALID_ARG, "unknown flags 0x%x", flags);
    const size_t need = chunk_bwd_workspace_bytes(T, num_seqs, Hk, Hv, dk, dv);
    if (!workspace || workspace_bytes < need)
        return fail(GDN_ERR_WORKSPACE, "workspace of %zu bytes < required %zu", workspace ? workspace_bytes : 0, need);
    if (reinterpret_cast<uintptr_t>(workspace) & 255u)
        return fail(GDN_ERR_WORKSPACE, "workspace must be 256-byte aligned");
    if (T > 0) {
        if ((st = check_row(q, ldq, (int64_t)Hk * dk, "q")) != GDN_OK) return st;
        if ((st = check_row(k, ldk, (int64_t)Hk * dk, "k")) != GDN_OK) return st;
        if ((st = check_row(v, ldv, (int64_t)Hv * dv, "v")) != GDN_OK) return st;
        if (!g || !beta || !dout || !dq || !dk_ || !dv_ || !dg || !dbeta)
            return fail(GDN_ERR_INVALID_ARG, "g/beta/dout or a gradient output is NULL");
    }
    return launch_chunk_bwd(q, k, v, ldq, ldk, ldv, dtype, g, beta, h0, dout, dh_final, cu_seqlens, num_seqs, T,
                            Hk, Hv, dk, dv, scale, (flags & GDN_QK_L2NORM) ? 1 : 0, dq, dk_, dv_, dg, dbeta, dh0,
                            workspace, (cudaStream_t)stream);
}

// workspace of gdn_shard_bwd: plan words, segment list, per-segment M, N,
// start states, start-state gradients and end-state gradients, then the
// backward kernel's own workspace over the segments
struct ShardBwdLayout {
    size_t plan, cu_seg, seg_seq, M, N, S, B, D, bwd, total;
};
static ShardBwdLayout shard_bwd_layout(int T, int num_seqs, int P, int Hk, int Hv, int dk, int dv) {
    ShardBwdLayout L{};
    const int nmax = num_seqs + P;
    const size_t st = sizeof(float) * (size_t)nmax * Hv * dk * dv;
    size_t o = 0;
    L.plan = o; o += align256(sizeof(int32_t) * (size_t)gdn_cp_plan_words(num_seqs, P));
    L.cu_seg = o; o += align256(sizeof(int32_t) * (size_t)(nmax + 1));
    L.seg_seq = o; o += align256(sizeof(int32_t) * (size_t)nmax);
    L.M = o; o += align256(sizeof(float) * (size_t)nmax * Hv * dk * dk);
    L.N = o; o += align256(st);
    L.S = o; o += align256(st);
    L.B = o; o += align256(st);
    L.D = o; o += align256(st);
    L.bwd = o; o += align256(chunk_bwd_workspace_bytes(T, nmax, Hk, Hv, dk, dv));
    L.total = o;
    return L;
}

size_t gdn_shard_bwd_workspace_size(int32_t T, int32_t num_seqs, int32_t n_shards, int32_t Hk, int32_t Hv,
                                    int32_t dk, int32_t dv) {
    if (T < 0 || num_seqs < 1 || n_shards < 1 || Hk < 1 || Hv < 1 || !dim_ok(dk) || !dim_ok(dv)) return 0;
    return shard_bwd_layout(T, num_seqs, n_shards, Hk, Hv, dk, dv).total;
}

gdn_status gdn_shard_bwd(const void* q, const void* k, const void* v, int64_t ldq, int64_t ldk, int64_t ldv,
                         gdn_dtype dtype, const float* g, const void* beta, const float* h0, const void* dout,
                         const float* dh_final, const int32_t* cu_seqlens, int32_t num_seqs, int32_t T, int32_t Hk,
                         int32_t Hv, int32_t dk, int32_t dv, float scale, uint32_t flags, int32_t n_shards,
                         float* dq, float* dk_, float* dv_, float* dg, float* dbeta, float* dh0, void* workspace,
                         size_t workspace_bytes, int32_t* plan_out, void* stream) {
    gdn_status st = check_heads(dtype, T, num_seqs, Hk, Hv, dk, dv);
    if (st != GDN_OK) return st;
    const int P = n_shards;
    if (P < 1 || P > 65536) return fail(GDN_ERR_INVALID_ARG, "n_shards=%d", P);
    if (T % P != 0) return fail(GDN_ERR_NOT_DIVISIBLE, "T=%d is not a multiple of n_shards=%d", T, P);
    if (!cu_seqlens || !dh0) return fail(GDN_ERR_INVALID_ARG, "cu_seqlens/dh0 is NULL");
    if (flags & ~(uint32_t)GDN_QK_L2NORM) return fail(GDN_ERR_INVALID_ARG, "unknown flags 0x%x", flags);
    const ShardBwdLayout L = shard_bwd_layout(T, num_seqs, P, Hk, Hv, dk, dv);
    if (!workspace || workspace_bytes < L.total)
        return fail(GDN_ERR_WORKSPACE, "workspace of %zu bytes < required %zu", workspace ? workspace_bytes : 0,
                    L.total);
    if (reinterpret_cast<uintptr_t>(workspace) & 255u) return fail(GDN_ERR_WORKSPACE, "workspace must be 256-byte aligned");
    if (T > 0) {
        if ((st = check_row(q, ldq, (int64_t)Hk * dk, "q")) != GDN_OK) return st;
        if ((st = check_row(k, ldk, (int64_t)Hk * dk, "k")) != GDN_OK) return st;
        if ((st = check_row(v, ldv, (int64_t)Hv * dv, "v")) != GDN_OK) return st;
        if (!g || !beta || !dout || !dq || !dk_ || !dv_ || !dg || !dbeta)
            return fail(GDN_ERR_INVALID_ARG, "g/beta/dout or a gradient output is NULL");
    }
    cudaStream_t s = (cudaStream_t)stream;
    const int l2 = (flags & GDN_QK_L2NORM) ? 1 : 0;
    unsigned char* w = static_cast<unsigned char*>(workspace);
    int32_t* plan = plan_out ? plan_out : reinterpret_cast<int32_t*>(w + L.plan);
    int32_t* cu_seg = reinterpret_cast<int32_t*>(w + L.cu_seg);
    int32_t* seg_seq = reinterpret_cast<int32_t*>(w + L.seg_seq);
    float* Ms = reinterpret_cast<float*>(w + L.M);
    float* Ns = reinterpret_cast<float*>(w + L.N);
    float* Ss = reinterpret_cast<float*>(w + L.S);
    float* Bs = reinterpret_cast<float*>(w + L.B);
    float* Ds = reinterpret_cast<float*>(w + L.D);
    void* bws = w + L.bwd;
    const int nmax = num_seqs + P;
    // 1. the segments: the shard plan's local segments of all shards
    if ((st = launch_plan(cu_seqlens, num_seqs, P, plan, s)) != GDN_OK) return st;
    if ((st = launch_segments(plan, num_seqs, P, T, nmax, cu_seg, seg_seq, s)) != GDN_OK) return st;
    // 2. every segment's affine state map (M, N) and its start state
    ChunkParams p{};
    p.q = k; p.k = k; p.v = v; p.ldq = ldk; p.ldk = ldk; p.ldv = ldv;
    p.g = g; p.beta = beta; p.cu = cu_seg;
    p.num_seqs = nmax; p.T = T; p.Hk = Hk; p.Hv = Hv; p.dk = dk; p.dv = dv;
    p.scale = 1.f; p.flags = flags; p.sumN = Ns; p.sumM = Ms;
    p.col_tile = chunk_col_tile(dtype, dk, dv);
    set_token_major(p);
    if ((st = launch_chunk(p, dtype, JOBS_SUMMARY, dim3(nmax, Hv, (dv + dk) / p.col_tile), s)) != GDN_OK) return st;
    if ((st = launch_seg_merge(true, plan, seg_seq, nmax, num_seqs, Hv, dk, dv, Ms, Ns, h0, Ss, s)) != GDN_OK)
        return st;
    // 3. each segment's start-state gradient from its own outputs (end gradient 0)
    if ((st = launch_chunk_bwd(q, k, v, ldq, ldk, ldv, dtype, g, beta, Ss, dout, nullptr, cu_seg, nmax, T, Hk, Hv,
                               dk, dv, scale, l2, dq, dk_, dv_, dg, dbeta, Bs, bws, s)) != GDN_OK)
        return st;
    // 4. the end-state gradients, each sequence's segments in reverse order
    if ((st = launch_seg_merge(false, plan, seg_seq, nmax, num_seqs, Hv, dk, dv, Ms, Bs, dh_final, Ds, s)) != GDN_OK)
        return st;
    // 5. the input gradients of every segment, from its true start state and end-state gradient
    if ((st = launch_chunk_bwd(q, k, v, ldq, ldk, ldv, dtype, g, beta, Ss, dout, Ds, cu_seg, nmax, T, Hk, Hv, dk,
                               dv, scale, l2, dq, dk_, dv_, dg, dbeta, Bs, bws, s)) != GDN_OK)
        return st;
    return launch_seg_dh0(plan, seg_seq, nmax, num_seqs, Hv, dk, dv, Bs, dh_final, dh0, s);
}

gdn_status gdn_chunk_fwd_heads(const void* q, const void* k, const void* v, gdn_dtype dtype, const float* g,
                               const void* beta, const float* h0, const int32_t* cu_seqlens, int32_t num_seqs,
                               int32_t T, int32_t Hk, int32_t Hv, int32_t dk, int32_t dv, float scale,
                               uint32_t flags, void* o, float* h_final, void* workspace, size_t workspace_bytes,
                               void* stream) {
    gdn_status st = check_heads(dtype, T, num_seqs, Hk, Hv, dk, dv);
    if (st != GDN_OK) return st;
    if (!cu_seqlens) return fail(GDN_ERR_INVALID_ARG, "cu_seqlens is NULL");
    const size_t need = gdn_chunk_fwd_workspace_size(num_seqs, Hv, dk, dv, dtype);
    if (workspace && workspace_bytes < need)
        return fail(GDN_ERR_WORKSPACE, "workspace of %zu bytes < required %zu", workspace_bytes, need);
    if (workspace && !al16(workspace)) return fail(GDN_ERR_WORKSPACE, "workspace must be 16-byte aligned");
    if (T > 0) {
        if (!q || !k || !v || !g || !beta || !o) return fail(GDN_ERR_INVALID_ARG, "q/k/v/g/beta/o is NULL");
        if (!al16(q) || !al16(k) || !al16(v) || !al16(o))
            return fail(GDN_ERR_INVALID_ARG, "q, k, v and o must be 16-byte aligned");
    }
    if (h_final && (reinterpret_cast<uintptr_t>(h_final) & 7u))
        return fail(GDN_ERR_INVALID_ARG, "h_final must be 8-byte aligned");
    ChunkParams p{};
    p.q = q; p.k = k; p.v = v; p.ldq = dk; p.ldk = dk; p.ldv = dv;
    p.g = g; p.beta = beta; p.h0 = h0; p.cu = cu_seqlens;
    p.num_seqs = num_seqs; p.T = T; p.Hk = Hk; p.Hv = Hv; p.dk = dk; p.dv = dv;
    p.scale = scale; p.flags = flags; p.o = o; p.h_final = h_final;
    p.col_tile = chunk_col_tile(dtype, dk, dv);
    // dense head-major [H, T, d]: a head is T rows further on
    p.hsq = p.hsk = (int64_t)T * dk;
    p.hsv = (int64_t)T * dv;
    p.ldo = dv;
    p.hso = (int64_t)T * dv;
    p.head_major = 1;
    if (workspace && T > 0 && chunk_tc_eligible(dtype, dk, dv)) p.sched = static_cast<int32_t*>(workspace);
    dim3 grid(num_seqs, Hv, dv / p.col_tile);
    return launch_chunk(p, dtype, JOBS_SEQS, grid, (cudaStream_t)stream);
}

gdn_status gdn_to_head_major(const void* x, int64_t ldx, gdn_dtype dtype, int32_t T, int32_t H, int32_t d,
                             void* y, void* stream) {
    if (dtype != GDN_F32 && dtype != GDN_BF16) return fail(GDN_ERR_DTYPE, "unknown dtype %d", (int)dtype);
    if (T < 0 || H < 1 || d < 1) return fail(GDN_ERR_INVALID_ARG, "T=%d H=%d d=%d", T, H, d);
    if ((d * (dtype == GDN_BF16 ? 2 : 4)) % 16 != 0) return fail(GDN_ERR_UNSUPPORTED_SHAPE, "d=%d rows not 16-byte", d);
    if (T == 0) return GDN_OK;
    if (!x || !y || !al16(x) || !al16(y)) return fail(GDN_ERR_INVALID_ARG, "x and y must be 16-byte aligned");
    if (ldx < (int64_t)H * d || (ldx * (dtype == GDN_BF16 ? 2 : 4)) % 16 != 0)
        return fail(GDN_ERR_INVALID_ARG, "token stride %lld of x", (long long)ldx);
    return launch_relayout(x, y, T, H, d, ldx, dtype, true, (cudaStream_t)stream);
}

gdn_status gdn_to_token_major(const void* y, gdn_dtype dtype, int32_t T, int32_t H, int32_t d, void* x,
                              int64_t ldx, void* stream) {
    if (dtype != GDN_F32 && dtype != GDN_BF16) return fail(GDN_ERR_DTYPE, "unknown dtype %d", (int)dtype);
    if (T < 0 || H < 1 || d < 1) return fail(GDN_ERR_INVALID_ARG, "T=%d H=%d d=%d", T, H, d);
    if ((d * (dtype == GDN_BF16 ? 2 : 4)) % 16 != 0) return fail(GDN_ERR_UNSUPPORTED_SHAPE, "d=%d rows not 16-byte", d);
    if (T == 0) return GDN_OK;
    if (!x || !y || !al16(x) || !al16(y)) return fail(GDN_ERR_INVALID_ARG, "x and y must be 16-byte aligned");
    if (ldx < (int64_t)H * d || (ldx * (dtype == GDN_BF16 ? 2 : 4)) % 16 != 0)
        return fail(GDN_ERR_INVALID_ARG, "token stride %lld of x", (long long)ldx);
    return launch_relayout(y, x, T, H, d, ldx, dtype, false, (cudaStream_t)stream);
}

size_t gdn_chunk_fwd_workspace_size(int32_t num_seqs, int32_t Hv, int32_t dk, int32_t dv, gdn_dtype dtype) {
    if (num_seqs < 1 || Hv < 1 || dk < 1 || dv < 1) return 0;
    const int tiles = dv / chunk_col_tile(dtype, dk, dv);
    return align256(sizeof(int32_t) * chunk_sched_words(num_seqs, Hv * (tiles > 0 ? tiles : 1)));
}

gdn_status gdn_chunk_summary(const void* k, const void* v, int64_t ldk, int64_t ldv, gdn_dtype dtype,
                             const float* g, const void* beta, const int32_t* cu_seqlens,
                             int32_t num_seqs, int32_t T, int32_t Hk, int32_t Hv, int32_t dk,
                             int32_t dv, uint32_t flags, float* M, float* N, void* stream) {
    gdn_status st = check_heads(dtype, T, num_seqs, Hk, Hv, dk, dv);
    if (st != GDN_OK) return st;
    if (!cu_seqlens || !M || !N) return fail(GDN_ERR_INVALID_ARG, "cu_seqlens/M/N is NULL");
    if ((reinterpret_cast<uintptr_t>(M) | reinterpret_cast<uintptr_t>(N)) & 7u)
        return fail(GDN_ERR_INVALID_ARG, "M and N must be 8-byte aligned");
    if (T > 0) {
        if ((st = check_row(k, ldk, (int64_t)Hk * dk, "k")) != GDN_OK) return st;
        if ((st = check_row(v, ldv, (int64_t)Hv * dv, "v")) != GDN_OK) return st;
        if (!g || !beta) return fail(GDN_ERR_INVALID_ARG, "g/beta is NULL");
    }
    ChunkParams p{};
    p.q = k; p.k = k; p.v = v; p.ldq = ldk; p.ldk = ldk; p.ldv = ldv;
    p.g = g; p.beta = beta; p.cu = cu_seqlens;
    p.num_seqs = num_seqs; p.T = T; p.Hk = Hk; p.Hv = Hv; p.dk = dk; p.dv = dv;
    p.scale = 1.f; p.flags = flags; p.sumN = N; p.sumM = M;
    p.col_tile = chunk_col_tile(dtype, dk, dv);
    set_token_major(p);
    dim3 grid(num_seqs, Hv, (dv + dk) / p.col_tile);
    return launch_chunk(p, dtype, JOBS_SUMMARY, grid, (cudaStream_t)stream);
}

gdn_status gdn_state_combine(const float* M, const float* N, const float* S0, int32_t P, int32_t Hv,
                             int32_t dk, int32_t dv, float* S_in, void* stream) {
    if (!M || !N || !S_in) return fail(GDN_ERR_INVALID_ARG, "M/N/S_in is NULL");
    if (!al16(M)) return fail(GDN_ERR_INVALID_ARG, "M must be 16-byte aligned");
    if (P < 1 || Hv < 1 || Hv > 65535) return fail(GDN_ERR_INVALID_ARG, "P=%d Hv=%d", P, Hv);
    if (!dim_ok(dk) || !dim_ok(dv))
        return fail(GDN_ERR_UNSUPPORTED_SHAPE, "dk=%d dv=%d must be in {32,64,128}", dk, dv);
    return launch_combine(M, N, S0, P, Hv, dk, dv, S_in, nullptr, (cudaStream_t)stream);
}

// pass-1 work order: ticket, entry count, one flag per (item, head, tile), sorted entries
static size_t pass1_sched_bytes(int num_seqs, int P, int Hv, int dk, int dv, gdn_dtype dtype) {
    const int tiles = (dv + dk) / chunk_col_tile(dtype, dk, dv);
    return align256(sizeof(int32_t) * chunk_sched_words(num_seqs + P, Hv * tiles));
}

size_t gdn_shard_fwd_workspace_size(int32_t T, int32_t num_seqs, int32_t n_shards, int32_t Hk,
                                    int32_t Hv, int32_t dk, int32_t dv, gdn_dtype dtype) {
    const size_t need = gdn::shard_fwd_workspace_min(T, num_seqs, n_shards, Hk, Hv, dk, dv, dtype);
    if (need == 0) return 0;
    const int P = gdn::internal_shards(T, num_seqs, n_shards, Hv, dk, dv, dtype);
    const bool mk = gdn::mchain_eligible(dtype, dk, dv) && P > 1 && T > 0;
    return need + (mk ? gdn::mchain_scratch_bytes(T, P, Hv) : 0);
}

size_t gdn_shard_fwd_workspace_min_size(int32_t T, int32_t num_seqs, int32_t n_shards, int32_t Hk,
                                        int32_t Hv, int32_t dk, int32_t dv, gdn_dtype dtype) {
    return gdn::shard_fwd_workspace_min(T, num_seqs, n_shards, Hk, Hv, dk, dv, dtype);
}

}  // extern "C"

namespace gdn {
// the workspace without the stored summary operands (the M chains then run in
// the chunk kernel, as the M half of each summary)
size_t shard_fwd_workspace_min(int32_t T, int32_t num_seqs, int32_t n_shards, int32_t Hk, int32_t Hv, int32_t dk,
                               int32_t dv, gdn_dtype dtype) {
    if (T < 0 || num_seqs < 1 || n_shards < 1 || Hk < 1 || Hv < 1 || dk < 1 || dv < 1) return 0;
    const int P = internal_shards(T, num_seqs, n_shards, Hv, dk, dv, dtype);
    const size_t cch = 2 * (size_t)Hk * dk + (size_t)Hv * dv;
    const size_t carry = (size_t)P * Hv * dk;
    return align256(sizeof(int32_t) * (size_t)gdn_cp_plan_words(num_seqs, P)) +
           align256((size_t)T * cch * esize(dtype)) +
           2 * align256(carry * dv * sizeof(float)) +  // carry N, S_in
           align256(carry * dk * sizeof(float)) +      // carry M
           pass1_sched_bytes(num_seqs, P, Hv, dk, dv, dtype);
}

// The layer's extras around the path: gates from the raw projections and the
// gated RMS norm of the output (null: gdn_shard_fwd's g / beta, plain o).
struct LayerExtras {
    const void* a;
    const float* A_log;
    const float* dt_bias;
    const void* z;  // or null: no norm
    int64_t ldz;
    const void* norm_w;
    float norm_eps;
};

static gdn_status shard_fwd_core(const void* x, const void* conv_w, const void* conv_b, int32_t conv_k,
                                 const float* g, const void* beta, const float* h0,
                                 const int32_t* cu_seqlens, int32_t num_seqs, int32_t T, int32_t Hk,
                                 int32_t Hv, int32_t dk, int32_t dv, float scale, uint32_t flags,
                                 int32_t n_shards, gdn_dtype dtype, void* workspace, size_t workspace_bytes,
                                 void* o, float* h_final, int32_t* plan_out, void* stream,
                                 const LayerExtras* ex) {
    gdn_status st = check_heads(dtype, T, num_seqs, Hk, Hv, dk, dv);
    if (st != GDN_OK) return st;
    if (n_shards < 1 || n_shards > 65536)
        return fail(GDN_ERR_INVALID_ARG, "n_shards=%d not in [1, 65536]", n_shards);
    if (T < n_shards) return fail(GDN_ERR_INVALID_ARG, "T=%d < n_shards=%d", T, n_shards);
    if (T % n_shards != 0)
        return fail(GDN_ERR_NOT_DIVISIBLE, "T=%d is not divisible by n_shards=%d", T, n_shards);
    if (conv_k < 1 || conv_k > 4) return fail(GDN_ERR_UNSUPPORTED_SHAPE, "conv_k=%d not in 1..4", conv_k);
    if (n_shards > 1 && T / n_shards < conv_k - 1)
        return fail(GDN_ERR_SHARD_TOO_SHORT, "shard length %d < conv halo %d", T / n_shards, conv_k - 1);
    if (!x || !conv_w || (!g && !ex) || !beta || !cu_seqlens || !o)
        return fail(GDN_ERR_INVALID_ARG, "x/conv_w/g/beta/cu_seqlens/o is NULL");
    if (ex) {
        if (!ex->a || !ex->A_log || !ex->dt_bias)
            return fail(GDN_ERR_INVALID_ARG, "a/A_log/dt_bias is NULL");
        if (ex->z) {
            if (!ex->norm_w || !al16(ex->z) || !al16(ex->norm_w))
                return fail(GDN_ERR_INVALID_ARG, "z and norm_w must be non-NULL and 16-byte aligned");
            if (ex->ldz < (int64_t)Hv * dv || ex->ldz % 8 != 0)
                return fail(GDN_ERR_INVALID_ARG, "row stride of z (%lld) must be >= Hv*dv and a multiple of 8",
                            (long long)ex->ldz);
            if (!(ex->norm_eps >= 0.f)) return fail(GDN_ERR_INVALID_ARG, "norm_eps must be >= 0");
        }
    }
    if (!al16(x) || !al16(o)) return fail(GDN_ERR_INVALID_ARG, "x and o must be 16-byte aligned");
    if (h_final && (reinterpret_cast<uintptr_t>(h_final) & 7u))
        return fail(GDN_ERR_INVALID_ARG, "h_final must be 8-byte aligned");
    const size_t need = shard_fwd_workspace_min(T, num_seqs, n_shards, Hk, Hv, dk, dv, dtype);
    if (!workspace || workspace_bytes < need)
        return fail(GDN_ERR_WORKSPACE, "workspace of %zu bytes < required %zu", workspace_bytes, need);
    // the shards the call runs on (the caller's, or finer for one long sequence)
    const int P = internal_shards(T, num_seqs, n_shards, Hv, dk, dv, dtype);
    // with room for the stored summary operands, the M chains run apart
    const size_t mk_bytes = mchain_eligible(dtype, dk, dv) && P > 1 ? mchain_scratch_bytes(T, P, Hv) : 0;
    const bool use_mk = mk_bytes > 0 && workspace_bytes >= need + mk_bytes && !(ex && ex->z) &&
                        (int64_t)P * Hv * ((T / P + 63) / 64) * 64 < ((int64_t)1 << 31);
    if (reinterpret_cast<uintptr_t>(workspace) & 255u)
        return fail(GDN_ERR_WORKSPACE, "workspace must be 256-byte aligned");
    cudaStream_t s = (cudaStream_t)stream;
    const int64_t cch = 2 * (int64_t)Hk * dk + (int64_t)Hv * dv;
    char* ws = static_cast<char*>(workspace);
    const int64_t words = gdn_cp_plan_words(num_seqs, P);
    int32_t* plan = reinterpret_cast<int32_t*>(ws);
    ws += align256(sizeof(int32_t) * (size_t)words);
    void* y = ws;
    ws += align256((size_t)T * cch * esize(dtype));
    const size_t carry = (size_t)P * Hv * dk;
    float* carryN = reinterpret_cast<float*>(ws);
    ws += align256(carry * dv * sizeof(float));
    float* S_in = reinterpret_cast<float*>(ws);
    ws += align256(carry * dv * sizeof(float));
    float* carryM = reinterpret_cast<float*>(ws);
    ws += align256(carry * dk * sizeof(float));
    int32_t* sched = reinterpret_cast<int32_t*>(ws);
    char* mk = static_cast<char*>(workspace) + need;  // stored summary operands (use_mk)

    auto mark = [&](int i) {
        if (i < g_phase_n) cudaEventRecord(g_phase_events[i], s);
    };
    mark(0);
    // 1. plan
    if ((st = launch_plan(cu_seqlens, num_seqs, P, plan, s)) != GDN_OK) return st;
    // 2. conv + SiLU, each shard reading its halo from the previous shard's rows
    if ((st = launch_conv(x, cch, dtype, T, (int)cch, conv_w, conv_b, conv_k, cu_seqlens, num_seqs,
                          nullptr, 0, y, cch, plan, P, s)) != GDN_OK)
        return st;
    mark(1);
    // 3. pass 1: every segment with a known initial state, plus [N | M] summaries
    ChunkParams p{};
    const size_t es = esize(dtype);
    p.q = y;
    p.k = static_cast<const char*>(y) + (size_t)Hk * dk * es;
    p.v = static_cast<const char*>(y) + (size_t)2 * Hk * dk * es;
    p.ldq = p.ldk = p.ldv = cch;
    p.g = g; p.beta = beta; p.h0 = h0; p.cu = cu_seqlens;
    p.num_seqs = num_seqs; p.T = T; p.Hk = Hk; p.Hv = Hv; p.dk = dk; p.dv = dv;
    p.scale = scale; p.flags = flags; p.o = o; p.h_final = h_final;
    p.sumN = carryN; p.sumM = carryM; p.S_in = S_in; p.plan = plan; p.n_shards = P;
    p.status = plan;  // an expired device wait is reported in the plan's status word
    const bool tc_norm = ex && ex->z && chunk_tc_eligible(dtype, dk, dv);
    if (ex) {
        p.a_raw = ex->a; p.A_log = ex->A_log; p.dt_bias = ex->dt_bias;
        if (tc_norm) { p.z = ex->z; p.ldz = ex->ldz; p.norm_w = ex->norm_w; p.norm_eps = ex->norm_eps; }
    }
    p.col_tile = chunk_col_tile(dtype, dk, dv);
    set_token_major(p);
    {
        if (chunk_tc_eligible(dtype, dk, dv)) p.sched = sched;  // filled by the order kernel
        if (use_mk) {
            const int nch = (T / P + 63) / 64;
            const size_t chunks = (size_t)P * Hv * nch, tile = chunks * 64 * 128 * es;
            p.m_external = 1;
            p.wk_nch = nch;
            p.wk_w = mk;
            p.wk_kt = mk + align256(tile);
            p.wk_eg = reinterpret_cast<float*>(mk + 2 * align256(tile));
        }
        // [N | M] column tiles; only the N tiles when the M chains run apart
        // (no work-queue tickets for M jobs that would be skipped)
        dim3 grid(num_seqs + P, Hv, (use_mk ? dv : dv + dk) / p.col_tile);
        if ((st = launch_chunk(p, dtype, JOBS_SHARD_PASS1, grid, s)) != GDN_OK) return st;
        p.sched = nullptr;
        if (use_mk) {  // the M halves of the summaries, from the operands the N halves stored
            if ((st = launch_mchain(plan, num_seqs, T, P, Hv, p.wk_w, p.wk_kt, p.wk_eg, carryM, s)) != GDN_OK)
                return st;
            p.m_external = 0;
            p.wk_w = p.wk_kt = nullptr;
            p.wk_eg = nullptr;
        }
    }
    mark(2);
    if (P > 1) {
        // 4. prefix merge of the shard carries
        if ((st = launch_combine(carryM, carryN, nullptr, P, Hv, dk, dv, S_in, plan, s)) != GDN_OK)
            return st;
        mark(3);
        // 5. pass 2: the first segment of every shard that continues a sequence
        // (the work queue's words are free again once pass 1 has run)
        if (chunk_tc_eligible(dtype, dk, dv)) p.sched = sched;
        dim3 grid(P, Hv, dv / p.col_tile);
        if ((st = launch_chunk(p, dtype, JOBS_SHARD_PASS2, grid, s)) != GDN_OK) return st;
        p.sched = nullptr;
    } else {
        mark(3);
    }
    if (ex && ex->z && !tc_norm) {  // kernels without the norm epilogue: a separate pass over o
        if ((st = launch_gated_norm(o, ex->z, ex->ldz, ex->norm_w, ex->norm_eps, T, Hv, dv, dtype, s)) != GDN_OK)
            return st;
    }
    mark(4);
    if (h_final) {
        if ((st = launch_empty_seq_final(cu_seqlens, num_seqs, Hv, dk, dv, h0, h_final, plan, s)) != GDN_OK)
            return st;
    }
    if (plan_out) {
        if (P != n_shards) {  // the caller's plan, with the status word of the call
            if ((st = launch_plan(cu_seqlens, num_seqs, n_shards, plan_out, s)) != GDN_OK) return st;
            if (cudaMemcpyAsync(plan_out, plan, sizeof(int32_t), cudaMemcpyDeviceToDevice, s) != cudaSuccess)
                return check_launch("plan status copy");
        } else if (cudaMemcpyAsync(plan_out, plan, sizeof(int32_t) * (size_t)words, cudaMemcpyDeviceToDevice,
                                   s) != cudaSuccess) {
            return check_launch("plan copy");
        }
    }
    mark(5);
    return GDN_OK;
}

}  // namespace gdn

extern "C" {

gdn_status gdn_shard_fwd(const void* x, const void* conv_w, const void* conv_b, int32_t conv_k,
                         const float* g, const void* beta, const float* h0,
                         const int32_t* cu_seqlens, int32_t num_seqs, int32_t T, int32_t Hk,
                         int32_t Hv, int32_t dk, int32_t dv, float scale, uint32_t flags,
                         int32_t n_shards, gdn_dtype dtype, void* workspace, size_t workspace_bytes,
                         void* o, float* h_final, int32_t* plan_out, void* stream) {
    return shard_fwd_core(x, conv_w, conv_b, conv_k, g, beta, h0, cu_seqlens, num_seqs, T, Hk, Hv, dk, dv, scale,
                          flags, n_shards, dtype, workspace, workspace_bytes, o, h_final, plan_out, stream, nullptr);
}

gdn_status gdn_layer_fwd(const void* x, const void* conv_w, const void* conv_b, int32_t conv_k, const void* a,
                         const void* b, const float* A_log, const float* dt_bias, const void* z, int64_t ldz,
                         const void* norm_w, float norm_eps, const float* h0, const int32_t* cu_seqlens,
                         int32_t num_seqs, int32_t T, int32_t Hk, int32_t Hv, int32_t dk, int32_t dv, float scale,
                         uint32_t flags, int32_t n_shards, gdn_dtype dtype, void* workspace,
                         size_t workspace_bytes, void* y, float* h_final, int32_t* plan_out, void* stream) {
    const LayerExtras ex{a, A_log, dt_bias, z, ldz, norm_w, norm_eps};
    return shard_fwd_core(x, conv_w, conv_b, conv_k, nullptr, b, h0, cu_seqlens, num_seqs, T, Hk, Hv, dk, dv,
                          scale, flags, n_shards, dtype, workspace, workspace_bytes, y, h_final, plan_out, stream,
                          &ex);
}

}  // extern "C"
