// Internal declarations shared by the CUDA translation units of libgdncp.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "gdn_cp.h"

namespace gdn {

constexpr int kChunk = 64;  // chunk size C of the WY/UT form

// ----------------------------------------------------------------------------
// host-side error reporting (api.cu)
// ----------------------------------------------------------------------------
gdn_status fail(gdn_status s, const char* fmt, ...);
gdn_status check_launch(const char* what);

// ----------------------------------------------------------------------------
// small device helpers
// ----------------------------------------------------------------------------
template <typename T> struct Elem;
template <> struct Elem<float> {
    static __device__ __forceinline__ float load(const float* p) { return *p; }
    static __device__ __forceinline__ float to_f(float x) { return x; }
    static __device__ __forceinline__ float from_f(float x) { return x; }
};
template <> struct Elem<__nv_bfloat16> {
    static __device__ __forceinline__ float load(const __nv_bfloat16* p) { return __bfloat162float(*p); }
    static __device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
    static __device__ __forceinline__ __nv_bfloat16 from_f(float x) { return __float2bfloat16_rn(x); }
};

// index of the last i in [0, n] with a[i] <= x (a non-decreasing, a[0] <= x)
__device__ __forceinline__ int upper_bound_minus1(const int32_t* a, int n, int x) {
    int lo = 0, hi = n;  // invariant: a[lo] <= x, answer in [lo, hi]
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if (__ldg(a + mid) <= x) lo = mid; else hi = mid - 1;
    }
    return lo;
}

// ----------------------------------------------------------------------------
// chunk kernels: one CTA runs one "job" = one token range of one value head
// and one tile of state columns, chunk after chunk.
// ----------------------------------------------------------------------------
struct ChunkJob {
    int t0, t1;            // tokens [t0, t1)
    int hv;                // value head
    int col0;              // first state column of this tile (within V or M)
    const float* init;     // initial state tile (row stride init_ld), or null = 0
    int64_t init_ld;
    float* fin;            // final state tile destination (row stride fin_ld), or null
    int64_t fin_ld;
    bool identity_init;    // M part of a summary: start from identity columns
    bool value_zero;       // M part of a summary: value columns are zero
    bool write_o;
    int wk_base;           // >= 0: the job stores its chunks' W rows, K~ and e^{G_last} from this chunk slot on
};

// Where a chunk kernel gets its jobs from.
enum JobSource : int {
    JOBS_SEQS = 0,        // gdn_chunk_fwd: grid (num_seqs, Hv, dv tiles)
    JOBS_SUMMARY = 1,     // gdn_chunk_summary: grid (num_seqs, Hv, (dv + dk) tiles)
    JOBS_SHARD_PASS1 = 2, // gdn_shard_fwd pass 1: grid (num_seqs + P, Hv, (dv + dk) tiles)
    JOBS_SHARD_PASS2 = 3  // gdn_shard_fwd pass 2: grid (P, Hv, dv tiles)
};

struct ChunkParams {
    const void* q; const void* k; const void* v;
    int64_t ldq, ldk, ldv;
    const float* g;
    const void* beta;
    const float* h0;
    const int32_t* cu;      // global cu_seqlens
    int num_seqs, T, Hk, Hv, dk, dv;
    float scale;
    uint32_t flags;
    void* o;                // [T, Hv, dv]
    float* h_final;         // [num_seqs, Hv, dk, dv] or null
    // summaries / shard path
    float* sumN;            // [n, Hv, dk, dv]
    float* sumM;            // [n, Hv, dk, dk]
    const float* S_in;      // [P, Hv, dk, dv]
    const int32_t* plan;    // plan words (shard path)
    int n_shards;
    int col_tile;           // state columns per CTA
    // work queue of the tcgen05 kernel (schedule words filled by the order
    // kernel, or null): the launch's items, (head, tile) pairs per item and
    // heads (the grid it stands for is items x heads x tiles); num_sms sizes
    // the schedule and the persistent grid
    int32_t* sched;
    int sched_items, sched_m, sched_ny;
    int num_sms;
    // device status word (plan or work-queue header) that receives
    // GDN_ERR_TIMEOUT when a bounded wait expires, or null
    int32_t* status;
    // limit of the split-item hand-over wait (ns of the global timer); a
    // test hook may also stop first halves from publishing their state
    long long handover_ns;
    int no_publish;
    // gates from the raw projections (a_raw != null): g = -exp(A_log[h])
    // softplus(a + dt_bias[h]) and beta = sigmoid(b), with b read through
    // `beta`; otherwise g and beta are read as given
    const void* a_raw;
    const float* A_log;
    const float* dt_bias;
    // head strides (elements) of q, k, v and the token / head strides of o:
    // token-major [T, H, d] has head stride d (o: token stride Hv*dv); the
    // head-major [H, T, d] layout has head stride T*d (o: token stride dv)
    int64_t hsq, hsk, hsv, ldo, hso;
    int head_major;  // q/k/v/o are head-major (the tensor-core kernel's TMA views)
    // gated RMS norm of the output (z != null, tensor-core kernel only):
    // o <- norm_w * o / sqrt(mean(o^2) + norm_eps) * silu(z), z row stride ldz
    const void* z;
    int64_t ldz;
    const void* norm_w;
    float norm_eps;
    // shard pass 1 with the M chains run apart (tensor-core kernel, bf16
    // d = 128): the N job of every spanning shard r stores, per chunk c of the
    // shard, its bf16 W rows and K~ tile ([slot * 64 rows x 128], slot =
    // (r * Hv + hv) * wk_nch + c) and e^{G_last} (wk_eg[slot]); the M jobs
    // are not run here
    void* wk_w;
    void* wk_kt;
    float* wk_eg;
    int wk_nch;
    int m_external;
};

// Token-major head strides (the layout every entry point but the head-major
// one uses).
inline void set_token_major(ChunkParams& p) {
    p.hsq = p.hsk = p.dk;
    p.hsv = p.dv;
    p.ldo = (int64_t)p.Hv * p.dv;
    p.hso = p.dv;
    p.head_major = 0;
}

// g and beta of token t, value head hv (E = the input dtype).  With raw
// projections, the wrappers' formulas ([HP-CP] P2P / all-gather forward):
// g = -exp(A_log) softplus(a + dt_bias) in fp32 (softplus(x) = x beyond 20,
// as torch's threshold), beta = sigmoid(b) rounded to the input dtype.
template <typename E>
__device__ __forceinline__ void gate_beta(const ChunkParams& p, int64_t t, int hv, float& g, float& b) {
    const int64_t i = t * p.Hv + hv;
    const E* bp = static_cast<const E*>(p.beta);
    if (p.a_raw) {
        const float x = Elem<E>::load(static_cast<const E*>(p.a_raw) + i) + __ldg(p.dt_bias + hv);
        const float sp = x > 20.f ? x : log1pf(__expf(x));
        g = -__expf(__ldg(p.A_log + hv)) * sp;
        b = Elem<E>::to_f(Elem<E>::from_f(1.f / (1.f + __expf(-Elem<E>::load(bp + i)))));
    } else {
        g = __ldg(p.g + i);
        b = Elem<E>::load(bp + i);
    }
}

// Resolve a block index (bx = job item, by = value head, bz = state tile)
// -> job.  Returns false when this CTA has nothing to do.
__device__ __forceinline__ bool make_job(const ChunkParams& p, int src, ChunkJob& j, int bx, int by, int bz) {
    const int hv = by;
    const int nvt = p.dv / p.col_tile;
    const int z = bz;
    j.hv = hv;
    j.identity_init = false;
    j.value_zero = false;
    j.wk_base = -1;
    j.init = nullptr;
    j.fin = nullptr;
    j.init_ld = p.dv;
    j.fin_ld = p.dv;
    auto clampT = [&](int t) { return t < 0 ? 0 : (t > p.T ? p.T : t); };
    if (src == JOBS_SEQS || src == JOBS_SUMMARY) {
        const int n = bx;
        j.t0 = clampT(__ldg(p.cu + n));
        j.t1 = clampT(__ldg(p.cu + n + 1));
        if (j.t1 < j.t0) j.t1 = j.t0;
        if (src == JOBS_SEQS) {
            j.col0 = z * p.col_tile;
            j.write_o = true;
            const int64_t st = ((int64_t)n * p.Hv + hv) * p.dk * p.dv + j.col0;
            if (p.h0) j.init = p.h0 + st;
            if (p.h_final) j.fin = p.h_final + st;
            return true;
        }
        j.write_o = false;
        if (z < nvt) {
            j.col0 = z * p.col_tile;
            j.fin = p.sumN + ((int64_t)n * p.Hv + hv) * p.dk * p.dv + j.col0;
        } else {
            j.col0 = (z - nvt) * p.col_tile;
            j.identity_init = true;
            j.value_zero = true;
            j.fin = p.sumM + ((int64_t)n * p.Hv + hv) * p.dk * p.dk + j.col0;
            j.fin_ld = p.dk;
        }
        return true;
    }
    // ---- shard path -------------------------------------------------------
    const int32_t* plan = p.plan;
    if (__ldg(plan) != 0) return false;  // malformed cu_seqlens: do nothing
    const int P = p.n_shards;
    const int part = p.T / P;
    const int64_t cu_base = 1 + (int64_t)P * GDN_PLAN_NFIELDS;
    if (src == JOBS_SHARD_PASS2) {
        const int r = bx;
        const int32_t* rec = plan + 1 + (int64_t)r * GDN_PLAN_NFIELDS;
        if (__ldg(rec + GDN_PLAN_IS_FIRST_RANK)) return false;
        if (z >= nvt) return false;
        const int32_t* lc = plan + cu_base + (int64_t)r * (p.num_seqs + 1);
        const int nloc = __ldg(rec + GDN_PLAN_LOCAL_NUM_SEQS);
        const int post = __ldg(rec + GDN_PLAN_POST_NUM_RANKS);
        const int n = __ldg(rec + GDN_PLAN_START_SEQ_IDX);
        j.t0 = r * part;
        j.t1 = r * part + __ldg(lc + 1);
        j.col0 = z * p.col_tile;
        j.write_o = true;
        j.init = p.S_in + ((int64_t)r * p.Hv + hv) * p.dk * p.dv + j.col0;
        const bool continues = (nloc == 1 && post > 0);
        if (!continues && p.h_final)
            j.fin = p.h_final + ((int64_t)n * p.Hv + hv) * p.dk * p.dv + j.col0;
        return true;
    }
    // pass 1: bx = flat (shard, local segment) slot
    const int slot = bx;
    int lo = 0, hi = P - 1;  // last shard with seg_offset <= slot
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if (__ldg(plan + 1 + (int64_t)mid * GDN_PLAN_NFIELDS + GDN_PLAN_SEG_OFFSET) <= slot) lo = mid;
        else hi = mid - 1;
    }
    const int r = lo;
    const int32_t* rec = plan + 1 + (int64_t)r * GDN_PLAN_NFIELDS;
    const int i = slot - __ldg(rec + GDN_PLAN_SEG_OFFSET);
    const int nloc = __ldg(rec + GDN_PLAN_LOCAL_NUM_SEQS);
    if (i < 0 || i >= nloc) return false;
    const int32_t* lc = plan + cu_base + (int64_t)r * (p.num_seqs + 1);
    const bool first_rank = __ldg(rec + GDN_PLAN_IS_FIRST_RANK) != 0;
    const int post = __ldg(rec + GDN_PLAN_POST_NUM_RANKS);
    const bool continues_in = (i == 0 && !first_rank);
    const bool continues_out = (i == nloc - 1 && post > 0);
    j.t0 = r * part + __ldg(lc + i);
    j.t1 = r * part + __ldg(lc + i + 1);
    const int64_t carry_st = ((int64_t)r * p.Hv + hv) * p.dk * p.dv;
    if (continues_in) {
        if (!continues_out) return false;       // only pass 2 for this segment
        // spanning shard: affine summary [N | M] from [0 | I]
        j.write_o = false;
        if (z < nvt) {
            j.col0 = z * p.col_tile;
            j.fin = p.sumN + carry_st + j.col0;
            if (p.m_external) j.wk_base = ((int)r * p.Hv + hv) * p.wk_nch;
        } else {
            if (p.m_external) return false;  // the M chain runs apart, from the stored operands
            j.col0 = (z - nvt) * p.col_tile;
            j.identity_init = true;
            j.value_zero = true;
            j.fin = p.sumM + ((int64_t)r * p.Hv + hv) * p.dk * p.dk + j.col0;
            j.fin_ld = p.dk;
        }
        return true;
    }
    if (z >= nvt) return false;
    // segment starts a sequence in this shard: initial state is known; its
    // global sequence from the plan's segment map (one load, no search)
    const int n = __ldg(plan + cu_base + (int64_t)(P + r) * (p.num_seqs + 1) + i);
    j.col0 = z * p.col_tile;
    j.write_o = true;
    const int64_t st = ((int64_t)n * p.Hv + hv) * p.dk * p.dv + j.col0;
    if (p.h0) j.init = p.h0 + st;
    if (continues_out) j.fin = p.sumN + carry_st + j.col0;  // constant carry (M = 0)
    else if (p.h_final) j.fin = p.h_final + st;
    return true;
}

__device__ __forceinline__ bool make_job(const ChunkParams& p, int src, ChunkJob& j) {
    return make_job(p, src, j, blockIdx.x, blockIdx.y, blockIdx.z);
}

// Tokens of job item x (the grid's x index) for the given job source; -1 if
// the item has no work.  Used to start the longest jobs first.
__device__ __forceinline__ int job_item_length(const ChunkParams& p, int src, int x) {
    if (src == JOBS_SEQS || src == JOBS_SUMMARY) {
        const int a = __ldg(p.cu + x), b = __ldg(p.cu + x + 1);
        return b > a ? b - a : 0;
    }
    const int32_t* plan = p.plan;
    if (__ldg(plan) != 0) return -1;
    const int P = p.n_shards;
    const int64_t cu_base = 1 + (int64_t)P * GDN_PLAN_NFIELDS;
    if (src == JOBS_SHARD_PASS2) {
        const int32_t* rec = plan + 1 + (int64_t)x * GDN_PLAN_NFIELDS;
        if (__ldg(rec + GDN_PLAN_IS_FIRST_RANK)) return -1;
        return __ldg(plan + cu_base + (int64_t)x * (p.num_seqs + 1) + 1);
    }
    int lo = 0, hi = P - 1;
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if (__ldg(plan + 1 + (int64_t)mid * GDN_PLAN_NFIELDS + GDN_PLAN_SEG_OFFSET) <= x) lo = mid;
        else hi = mid - 1;
    }
    const int32_t* rec = plan + 1 + (int64_t)lo * GDN_PLAN_NFIELDS;
    const int i = x - __ldg(rec + GDN_PLAN_SEG_OFFSET);
    if (i < 0 || i >= __ldg(rec + GDN_PLAN_LOCAL_NUM_SEQS)) return -1;
    const int32_t* lc = plan + cu_base + (int64_t)lo * (p.num_seqs + 1);
    return __ldg(lc + i + 1) - __ldg(lc + i);
}

// Longest-first block order.  The hardware starts CTAs roughly in linear
// block order, so the linear index L is mapped to (item of rank L / (heads *
// tiles), head, tile) with items ranked by decreasing length (ties by index).
// Cooperative over the CTA (all NT threads); len is shared scratch of
// kMaxLptItems ints.  Grids with more items keep the natural order.
constexpr int kMaxLptItems = 512;
template <int NT>
__device__ __forceinline__ void lpt_block(const ChunkParams& p, int src, int* len, int* pick, int& bx,
                                          int& by, int& bz) {
    const int S = gridDim.x;
    bx = blockIdx.x;
    by = blockIdx.y;
    bz = blockIdx.z;
    if (S > kMaxLptItems) return;
    for (int s = threadIdx.x; s < S; s += NT) len[s] = job_item_length(p, src, s);
    __syncthreads();
    const int64_t L = blockIdx.x + (int64_t)gridDim.x * (blockIdx.y + (int64_t)gridDim.y * blockIdx.z);
    const int per = gridDim.y * gridDim.z;
    const int r = (int)(L / per), rem = (int)(L % per);
    for (int n = threadIdx.x; n < S; n += NT) {
        const int ln = len[n];
        int rank = 0;
        for (int m = 0; m < S; ++m) {
            const int lm = len[m];
            rank += (lm > ln) || (lm == ln && m < n);
        }
        if (rank == r) *pick = n;
    }
    __syncthreads();
    bx = *pick;
    by = rem % gridDim.y;
    bz = rem / gridDim.y;
}

// Schedule words of a ticket-scheduled launch: [0] ticket counter, [1] entry
// count, [2] status word (0, or GDN_ERR_TIMEOUT once a bounded wait expired),
// [3] unused, then one hand-over flag per (item, head, tile) from
// kSchedHeader, then the sorted entries at an even offset (read as int2).
constexpr int kSchedHeader = 4;
__host__ __device__ __forceinline__ int64_t chunk_sched_order_off(int S, int m) {
    const int64_t o = kSchedHeader + (int64_t)S * m;
    return o + (o & 1);
}
// schedule.cu: words of a launch's schedule (S items, m head/tile pairs) and
// the kernel that fills them (zeroed ticket and flags, sorted entries)
inline size_t chunk_sched_words(int S, int m) { return (size_t)chunk_sched_order_off(S, m) + 4 * (size_t)S; }
// split rules of the order kernel: none, middle halves, short tails
constexpr int kSplitNone = 0, kSplitHalves = 1, kSplitTail = 2;
gdn_status launch_chunk_order(const ChunkParams& p, int src, int S, int m, int split_rule, cudaStream_t s);

// launchers (chunk_bf16.cu / chunk_f32.cu)
gdn_status launch_chunk_bf16(const ChunkParams& p, int src, dim3 grid, cudaStream_t s);
gdn_status launch_chunk_f32(const ChunkParams& p, int src, dim3 grid, cudaStream_t s);
// tcgen05 kernel (chunk_tc.cu): bf16 with d_k = d_v = 128, full-width state tiles
bool chunk_tc_eligible(gdn_dtype dt, int dk, int dv);
gdn_status launch_chunk_tc(ChunkParams p, int src, dim3 grid, cudaStream_t s);
// the M chains of the shard summaries run apart from their stored operands
// (csrc/mchain.cu): scratch bytes of the stored W rows, K~ and e^{G_last},
// then the segments' products when the chains are cut (0 for P < 2), and the
// launch over the plan's spanning shards into M [P, Hv, 128, 128]
bool mchain_eligible(gdn_dtype dt, int dk, int dv);
// gdn_shard_fwd's workspace without the stored summary operands
size_t shard_fwd_workspace_min(int32_t T, int32_t num_seqs, int32_t n_shards, int32_t Hk, int32_t Hv, int32_t dk,
                               int32_t dv, gdn_dtype dtype);
size_t mchain_scratch_bytes(int T, int P, int Hv);
gdn_status launch_mchain(const int32_t* plan, int num_seqs, int T, int P, int Hv, void* w, void* kt,
                         const float* eg, float* M, cudaStream_t s);
extern __device__ int g_gdn_timeouts;
int chunk_col_tile(gdn_dtype dt, int dk, int dv);

// plan.cu
gdn_status launch_plan(const int32_t* cu, int num_seqs, int P, int32_t* plan, cudaStream_t s);
// SMs of the current device (cached per device)
int device_sm_count();
// shards a gdn_shard_fwd call runs on (csrc/api.cu)
int internal_shards(int T, int num_seqs, int P, int Hv, int dk, int dv, gdn_dtype dtype);
// conv.cu: per-shard conv; plan == null -> one shard with an explicit halo
gdn_status launch_conv(const void* x, int64_t ldx, gdn_dtype dt, int T, int C, const void* w,
                       const void* b, int Kc, const int32_t* cu, int num_seqs, const void* halo,
                       int halo_len, void* y, int64_t ldy, const int32_t* plan, int P,
                       cudaStream_t s);
// combine.cu: plan == null -> every shard affine
gdn_status launch_combine(const float* M, const float* N, const float* S0, int P, int Hv, int dk,
                          int dv, float* S_in, const int32_t* plan, cudaStream_t s);
// layout.cu: [T, H, d] (token stride ld) <-> dense [H, T, d]
gdn_status launch_relayout(const void* src, void* dst, int64_t T, int H, int d, int64_t ld, gdn_dtype dt,
                           bool to_heads, cudaStream_t s);
// backward.cu: the backward of the recurrence over (sequence, value head) jobs
size_t chunk_bwd_workspace_bytes(int T, int num_seqs, int Hk, int Hv, int dk, int dv);
gdn_status launch_chunk_bwd(const void* q, const void* k, const void* v, int64_t ldq, int64_t ldk, int64_t ldv,
                            gdn_dtype dtype, const float* g, const void* beta, const float* h0, const void* dout,
                            const float* dh_final, const int32_t* cu, int num_seqs, int T, int Hk, int Hv, int dk,
                            int dv, float scale, int l2, float* dq, float* dk_, float* dv_, float* dg, float* dbeta,
                            float* dh0, void* workspace, cudaStream_t s);
// shard_bwd.cu: segments of the shard plan, and the merges of the backward across shards
gdn_status launch_segments(const int32_t* plan, int num_seqs, int P, int T, int nmax, int32_t* cu_seg,
                           int32_t* seg_seq, cudaStream_t s);
gdn_status launch_seg_merge(bool fwd, const int32_t* plan, const int32_t* seg_seq, int nmax, int num_seqs, int Hv,
                            int dk, int dv, const float* M, const float* NB, const float* init, float* out,
                            cudaStream_t s);
gdn_status launch_seg_dh0(const int32_t* plan, const int32_t* seg_seq, int nmax, int num_seqs, int Hv, int dk,
                          int dv, const float* dh0_seg, const float* dh_final, float* dh0, cudaStream_t s);
// gated RMS norm of o in place (combine.cu), for the kernels without the epilogue
gdn_status launch_gated_norm(void* o, const void* z, int64_t ldz, const void* w, float eps, int64_t T, int Hv,
                             int dv, gdn_dtype dt, cudaStream_t s);
// empty sequences in the shard path: h_final = h0 or 0
gdn_status launch_empty_seq_final(const int32_t* cu, int num_seqs, int Hv, int dk, int dv,
                                  const float* h0, float* h_final, const int32_t* plan,
                                  cudaStream_t s);

}  // namespace gdn
