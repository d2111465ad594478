// Backward of the gated delta rule (hyper-parallel page
// linear_attention_context_parallel.py: the state gradient that
// _RecvInitialStateP2PFunction / _SendFinalStateP2PFunction send back the
// other way; the recurrence is the one _run_prepared_gdn_chunks computes in
// chunked form).
//
// Per token, with a = e^g, P = a S_prev, u = v - P^T k, S = P + beta k u^T and
// o = S^T (scale q), reverse mode with the state gradient dS walks the tokens
// backwards:
//   dq = scale (P do + beta k (u . do));   dS += scale q do^T
//   dbeta = k . (dS u);   du = beta dS^T k;   dv = du
//   dS -= k du^T  (= dP);  dk = beta dS_before u - P du;   dg = <P, dP>;  dS = a dP
// (q, k are the L2-normalised vectors when the flag is set; their gradients
// go back through x / sqrt(|x|^2 + 1e-6) in a last pass.)
//
// One CTA of 512 threads runs one (sequence, value head) job.  Thread (row
// r, lane lr of the row) holds S[r][lr + TPR i], i < CPT, in registers and
// the same elements of dS in shared memory (thread-interleaved, no bank
// conflicts).  Row sums (K-vectors) reduce over the TPR lanes
// of a row by shuffles; column sums (V-vectors) over the rows through shared
// memory.  The states before each token are recomputed: a forward pass over
// the job (threads owning state columns, so that its column sums need no
// block-wide sync) keeps the state at every 8-token block start in the
// workspace; going backwards, each block is replayed once (row-owning, as
// the reverse step) to keep the state before each of its tokens (a per-job
// scratch of 8 states, small enough to stay in L2) and its u = v - P^T k.
// Each 64-token chunk's q, k, v, do, g and beta are staged in shared memory.
#include "gdn_internal.cuh"

namespace gdn {
namespace {

constexpr int NTB = 512;  // threads per CTA
constexpr int NWB = NTB / 32;
constexpr int kSub = 8;   // tokens per replayed block

struct BwdParams {
    const void* q; const void* k; const void* v;
    int64_t ldq, ldk, ldv;
    const float* g;
    const void* beta;
    const float* h0;
    const void* dout;        // [T, Hv, dv]
    const float* dh_final;   // [N, Hv, dk, dv] or null
    const int32_t* cu;
    int num_seqs, T, Hk, Hv, dk, dv;
    float scale;
    int l2;
    const float* rq;         // [T, Hk] 1/|q| (l2) or null
    const float* rk;
    float* dq; float* dk_; float* dv_; float* dg; float* dbeta; float* dh0;
    float* ckpt;             // block-start states, slot (cu[n] / 8 + n + b) per sequence n
    float* scratch;          // per job: the states before the tokens of one block
};

// 1 / sqrt(|x|^2 + 1e-6) of every (token, q/k head) row of q and k; one warp per row
template <typename E>
__global__ void bwd_norms_kernel(const E* __restrict__ q, const E* __restrict__ k, int64_t ldq, int64_t ldk,
                                 int T, int Hk, int dk, float* __restrict__ rq, float* __restrict__ rk) {
    const int w = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
    if (w >= T * Hk) return;
    const int t = w / Hk, h = w - t * Hk;
    float sq = 0.f, sk = 0.f;
    for (int i = lane; i < dk; i += 32) {
        const float a = Elem<E>::load(q + (int64_t)t * ldq + (int64_t)h * dk + i);
        const float b = Elem<E>::load(k + (int64_t)t * ldk + (int64_t)h * dk + i);
        sq = fmaf(a, a, sq);
        sk = fmaf(b, b, sk);
    }
#pragma unroll
    for (int off = 16; off; off >>= 1) {
        sq += __shfl_xor_sync(0xffffffffu, sq, off);
        sk += __shfl_xor_sync(0xffffffffu, sk, off);
    }
    if (lane == 0) {
        rq[w] = rsqrtf(sq + 1e-6f);
        rk[w] = rsqrtf(sk + 1e-6f);
    }
}

// dx = r dxn - r^3 (x . dxn) x in place over the gradient rows of q and k
template <typename E>
__global__ void bwd_l2_kernel(const E* __restrict__ q, const E* __restrict__ k, int64_t ldq, int64_t ldk,
                              int T, int Hk, int dk, const float* __restrict__ rq, const float* __restrict__ rk,
                              float* __restrict__ dq, float* __restrict__ dkk) {
    const int w = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
    if (w >= 2 * T * Hk) return;
    const bool isk = w >= T * Hk;
    const int row = isk ? w - T * Hk : w;
    const int t = row / Hk, h = row - t * Hk;
    const E* x = (isk ? k + (int64_t)t * ldk : q + (int64_t)t * ldq) + (int64_t)h * dk;
    float* d = (isk ? dkk : dq) + (int64_t)row * dk;
    const float r = isk ? rk[row] : rq[row];
    float xd = 0.f;
    for (int i = lane; i < dk; i += 32) xd = fmaf(Elem<E>::load(x + i), d[i], xd);
#pragma unroll
    for (int off = 16; off; off >>= 1) xd += __shfl_xor_sync(0xffffffffu, xd, off);
    const float c = r * r * r * xd;
    for (int i = lane; i < dk; i += 32) d[i] = r * d[i] - c * Elem<E>::load(x + i);
}

// One (sequence, value head) job per CTA.  Thread (row, lr): TPR threads per
// state row, thread lr of a row owning the CPT columns lr + TPR i (strided, so
// that the lanes of a warp read consecutive words of a staged row).
template <typename E, int DK, int DV>
struct BwdJob {
    static constexpr int TPR = NTB / DK;
    static constexpr int CPT = DV / TPR;
    static_assert(TPR >= 1 && TPR <= 32 && (32 % TPR) == 0 && CPT >= 1 && DV % TPR == 0, "shape");
    // the forward steps own columns instead: TPC threads per state column,
    // thread rb of a column holding the RPT rows rb RPT .. rb RPT + RPT
    static constexpr int TPC = NTB / DV;
    static constexpr int RPT = DK / TPC;
    static_assert(TPC >= 1 && TPC <= 32 && (32 % TPC) == 0 && RPT == CPT, "shape");

    struct Smem {
        float ks[kChunk][DK], qs[kChunk][DK];
        float vs[kChunk][DV], dos[kChunk][DV];
        float gs[kChunk], bs[kChunk], rks[kChunk], rqs[kChunk];
        float red[NWB][DV];
        float vec[DV];
        float sred[NWB][2];
        float us[kSub][DV];   // u = v - P^T k of the block's tokens, from the replay
        float dS[CPT][NTB];   // the state gradient, element i of thread t at [i][t]
    };

    const BwdParams& p;
    Smem& sm;
    const int tid, lane, warp, row, lr, ccol, rb;
    int n, hv, hk;

    __device__ BwdJob(const BwdParams& p_, Smem& sm_)
        : p(p_), sm(sm_), tid(threadIdx.x), lane(threadIdx.x & 31), warp(threadIdx.x >> 5),
          row(threadIdx.x / TPR), lr(threadIdx.x % TPR), ccol(threadIdx.x / TPC), rb(threadIdx.x % TPC) {}
    __device__ __forceinline__ int col(int i) const { return lr + TPR * i; }

    // sum over the rows of each of this thread's columns.  Within a warp the
    // lanes sharing a column block halve their values at each exchange
    // (each keeps the half its lane bit selects and adds the partner's copy),
    // so the warp's row sums end up spread over those lanes; then the warps'
    // sums go through shared memory.
    __device__ __forceinline__ void vred(float (&x)[CPT]) {
        int off_cols = 0;
#pragma unroll
        for (int off = TPR, half = CPT / 2; off < 32; off <<= 1, half >>= 1) {
            const bool hi = (lane & off) != 0;
#pragma unroll
            for (int i = 0; i < half; ++i) {
                const float send = hi ? x[i] : x[i + half];
                const float keep = hi ? x[i + half] : x[i];
                x[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
            }
            if (hi) off_cols += half;
        }
        constexpr int kept = CPT * TPR / 32;  // columns each lane holds at the end
#pragma unroll
        for (int i = 0; i < kept; ++i) sm.red[warp][col(off_cols + i)] = x[i];
        __syncthreads();
        if (tid < DV) {
            float s = 0.f;
#pragma unroll
            for (int w = 0; w < NWB; ++w) s += sm.red[w][tid];
            sm.vec[tid] = s;
        }
        __syncthreads();
#pragma unroll
        for (int i = 0; i < CPT; ++i) x[i] = sm.vec[col(i)];
    }
    // sum over the TPR threads of a row
    __device__ __forceinline__ float rred(float x) {
#pragma unroll
        for (int off = 1; off < TPR; off <<= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
        return x;
    }

    // kept states are thread-interleaved (element i of thread t at [i][t]):
    // every warp store and load covers 128 contiguous bytes
    __device__ __forceinline__ void store_state(float* base, int slot, const float (&s)[CPT]) {
        float* d = base + (int64_t)slot * CPT * NTB + tid;
#pragma unroll
        for (int i = 0; i < CPT; ++i) d[i * NTB] = s[i];
    }
    __device__ __forceinline__ void load_state(const float* base, int slot, float (&s)[CPT]) {
        const float* d = base + (int64_t)slot * CPT * NTB + tid;
#pragma unroll
        for (int i = 0; i < CPT; ++i) s[i] = __ldcg(d + i * NTB);
    }

    // the same layout addressed by (row, column), for the column-owning steps
    __device__ __forceinline__ static int64_t at(int r, int c) {
        return (int64_t)(c / TPR) * NTB + (int64_t)r * TPR + (c % TPR);
    }
    __device__ __forceinline__ void store_state_col(float* base, int slot, const float (&s)[RPT]) {
        float* d = base + (int64_t)slot * CPT * NTB;
#pragma unroll
        for (int j = 0; j < RPT; ++j) d[at(rb * RPT + j, ccol)] = s[j];
    }
    __device__ __forceinline__ void load_state_col(const float* base, int slot, float (&s)[RPT]) {
        const float* d = base + (int64_t)slot * CPT * NTB;
#pragma unroll
        for (int j = 0; j < RPT; ++j) s[j] = __ldcg(d + at(rb * RPT + j, ccol));
    }

    // tokens [tb, tb + cnt) of the job into shared memory
    __device__ void stage(int tb, int cnt, bool all) {
        __syncthreads();  // every thread is done with the previous chunk's tiles
        const E* q = static_cast<const E*>(p.q);
        const E* k = static_cast<const E*>(p.k);
        const E* v = static_cast<const E*>(p.v);
        const E* dout = static_cast<const E*>(p.dout);
        const E* beta = static_cast<const E*>(p.beta);
        for (int e = tid; e < cnt * DK; e += NTB) {
            const int j = e / DK, i = e - j * DK;
            const int64_t t = tb + j;
            sm.ks[j][i] = Elem<E>::load(k + t * p.ldk + (int64_t)hk * DK + i);
            if (all) sm.qs[j][i] = Elem<E>::load(q + t * p.ldq + (int64_t)hk * DK + i);
        }
        for (int e = tid; e < cnt * DV; e += NTB) {
            const int j = e / DV, i = e - j * DV;
            const int64_t t = tb + j;
            sm.vs[j][i] = Elem<E>::load(v + t * p.ldv + (int64_t)hv * DV + i);
            if (all) sm.dos[j][i] = Elem<E>::load(dout + (t * p.Hv + hv) * DV + i);
        }
        if (tid < cnt) {
            const int64_t t = tb + tid;
            sm.gs[tid] = p.g[t * p.Hv + hv];
            sm.bs[tid] = Elem<E>::load(beta + t * p.Hv + hv);
            sm.rks[tid] = p.l2 ? p.rk[t * p.Hk + hk] : 1.f;
            sm.rqs[tid] = p.l2 ? p.rq[t * p.Hk + hk] : 1.f;
        }
        __syncthreads();
    }

    // the same step row-owning (the replay: its states are stored in the
    // row-owning layout with whole-line stores); u of its columns to row 0's
    // threads, which keep it in shared memory for the reverse step
    __device__ __forceinline__ void fwd_step_rows(int j, float (&S)[CPT], float* us_row) {
        const float a = __expf(sm.gs[j]), b = sm.bs[j];
        const float kr = sm.ks[j][row] * sm.rks[j];
        float x[CPT];
#pragma unroll
        for (int i = 0; i < CPT; ++i) {
            S[i] *= a;
            x[i] = S[i] * kr;
        }
        vred(x);  // a S^T k
#pragma unroll
        for (int i = 0; i < CPT; ++i) {
            const float u = sm.vs[j][col(i)] - x[i];
            if (row == 0) us_row[col(i)] = u;
            S[i] = fmaf(b * kr, u, S[i]);
        }
    }

    // S <- a S + beta k (v - a S^T k)^T for staged token j, column-owning
    // (the column's sum over the rows is a shuffle among its TPC threads, no
    // block-wide sync); returns u = v - a S^T k of the thread's column
    __device__ __forceinline__ float fwd_step(int j, float (&S)[RPT]) {
        const float a = __expf(sm.gs[j]), b = sm.bs[j], rk = sm.rks[j];
        float kr[RPT];
        if constexpr (RPT % 4 == 0) {
            const float4* k4 = reinterpret_cast<const float4*>(&sm.ks[j][rb * RPT]);
#pragma unroll
            for (int q4 = 0; q4 < RPT / 4; ++q4) {
                const float4 f = k4[q4];
                kr[4 * q4] = f.x * rk;
                kr[4 * q4 + 1] = f.y * rk;
                kr[4 * q4 + 2] = f.z * rk;
                kr[4 * q4 + 3] = f.w * rk;
            }
        } else {
#pragma unroll
            for (int jj = 0; jj < RPT; ++jj) kr[jj] = sm.ks[j][rb * RPT + jj] * rk;
        }
        float x = 0.f;
#pragma unroll
        for (int jj = 0; jj < RPT; ++jj) {
            S[jj] *= a;
            x = fmaf(S[jj], kr[jj], x);
        }
#pragma unroll
        for (int off = 1; off < TPC; off <<= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
        const float u = sm.vs[j][ccol] - x;
#pragma unroll
        for (int jj = 0; jj < RPT; ++jj) S[jj] = fmaf(b * kr[jj], u, S[jj]);
        return u;
    }

    // the reverse step of staged token j (global token t), from the state
    // before it (Sp); the state gradient is in shared memory
    __device__ __forceinline__ void bwd_step(int j, int64_t t, const float (&Sp)[CPT]) {
        const float a = __expf(sm.gs[j]), b = sm.bs[j];
        const float kr = sm.ks[j][row] * sm.rks[j], qr = sm.qs[j][row] * sm.rqs[j] * p.scale;
        float x[CPT];
        float udo = 0.f, pdo = 0.f, dsu = 0.f;
#pragma unroll
        for (int i = 0; i < CPT; ++i) {
            const float u = sm.us[j % kSub][col(i)], dov = sm.dos[j][col(i)];
            udo = fmaf(u, dov, udo);
            pdo = fmaf(a * Sp[i], dov, pdo);
            const float ds = fmaf(qr, dov, sm.dS[i][tid]);  // dS += scale q do^T
            sm.dS[i][tid] = ds;
            dsu = fmaf(ds, u, dsu);
            x[i] = ds * kr;
        }
        udo = rred(udo);
        pdo = rred(pdo);
        dsu = rred(dsu);  // (dS u)[row]
        const float dqr = p.scale * (pdo + b * kr * udo);  // w.r.t. the normalised q
        vred(x);          // dS^T k
        float pdu = 0.f, pdp = 0.f;
        float* dv = p.dv_ + (t * p.Hv + hv) * DV;
#pragma unroll
        for (int i = 0; i < CPT; ++i) {
            const float du = b * x[i];
            if (row == 0) dv[col(i)] = du;
            const float ds = fmaf(-kr, du, sm.dS[i][tid]);  // dP
            pdu = fmaf(a * Sp[i], du, pdu);
            pdp = fmaf(a * Sp[i], ds, pdp);
            sm.dS[i][tid] = a * ds;
        }
        pdu = rred(pdu);
        if (lr == 0) {
            atomicAdd(p.dq + (t * p.Hk + hk) * DK + row, dqr);
            atomicAdd(p.dk_ + (t * p.Hk + hk) * DK + row, b * dsu - pdu);
        }
        // dbeta = k . (dS u), dg = <P, dP>
        float s1 = lr == 0 ? kr * dsu : 0.f, s2 = pdp;
#pragma unroll
        for (int off = 16; off; off >>= 1) {
            s1 += __shfl_xor_sync(0xffffffffu, s1, off);
            s2 += __shfl_xor_sync(0xffffffffu, s2, off);
        }
        if (lane == 0) {
            sm.sred[warp][0] = s1;
            sm.sred[warp][1] = s2;
        }
        __syncthreads();
        if (tid == 0) {
            float b1 = 0.f, b2 = 0.f;
#pragma unroll
            for (int w = 0; w < NWB; ++w) {
                b1 += sm.sred[w][0];
                b2 += sm.sred[w][1];
            }
            p.dbeta[t * p.Hv + hv] = b1;
            p.dg[t * p.Hv + hv] = b2;
        }
    }

    __device__ void run() {
        n = blockIdx.x;
        hv = blockIdx.y;
        hk = hv / (p.Hv / p.Hk);
        const int t0 = __ldg(p.cu + n), L = __ldg(p.cu + n + 1) - t0;
        const int nch = (L + kChunk - 1) / kChunk;
        const int64_t state = (int64_t)DK * DV;
        // block b (kSub tokens) of sequence n: slot t0 / kSub + n + b (never
        // overlaps the next sequence's)
        float* ck = p.ckpt + (int64_t)(t0 / kSub + n) * p.Hv * state + (int64_t)hv * state;
        const int ck_stride = p.Hv;  // in states, between consecutive blocks
        float* tok = p.scratch + ((int64_t)n * p.Hv + hv) * kSub * state;
        const int64_t sidx = ((int64_t)n * p.Hv + hv) * state + (int64_t)row * DV;
        // forward (column-owning): the state at every block start
        float S[RPT];
        const int64_t sidx_col = ((int64_t)n * p.Hv + hv) * state + (int64_t)rb * RPT * DV + ccol;
#pragma unroll
        for (int jj = 0; jj < RPT; ++jj) S[jj] = p.h0 ? p.h0[sidx_col + (int64_t)jj * DV] : 0.f;
        for (int c = 0; c < nch; ++c) {
            const int cnt = min(kChunk, L - c * kChunk);
            stage(t0 + c * kChunk, cnt, false);
            for (int j = 0; j < cnt; ++j) {
                if (j % kSub == 0) store_state_col(ck, (c * (kChunk / kSub) + j / kSub) * ck_stride, S);
                fwd_step(j, S);
            }
        }
        // backward
#pragma unroll
        for (int i = 0; i < CPT; ++i) sm.dS[i][tid] = p.dh_final ? p.dh_final[sidx + col(i)] : 0.f;
        for (int c = nch - 1; c >= 0; --c) {
            const int cnt = min(kChunk, L - c * kChunk), tb = t0 + c * kChunk;
            stage(tb, cnt, true);
            const int nb = (cnt + kSub - 1) / kSub;
            for (int bl = nb - 1; bl >= 0; --bl) {
                const int j0 = bl * kSub, j1 = min(cnt, j0 + kSub);
                float R[CPT];
                load_state(ck, (c * (kChunk / kSub) + bl) * ck_stride, R);
                for (int j = j0; j < j1; ++j) {  // the state before each token, and its u
                    store_state(tok, j - j0, R);
                    fwd_step_rows(j, R, sm.us[j - j0]);
                }
                __syncthreads();  // the block's u is visible to every thread
                for (int j = j1 - 1; j >= j0; --j) {
                    float Sp[CPT];
                    load_state(tok, j - j0, Sp);
                    bwd_step(j, tb + j, Sp);
                }
            }
        }
        __syncthreads();
#pragma unroll
        for (int i = 0; i < CPT; ++i) p.dh0[sidx + col(i)] = sm.dS[i][tid];
    }
};

template <typename E, int DK, int DV>
__global__ void __launch_bounds__(NTB, 1) bwd_job_kernel(const BwdParams p) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    using J = BwdJob<E, DK, DV>;
    J job(p, *reinterpret_cast<typename J::Smem*>(smem_raw));
    job.run();
}

}  // namespace

gdn_status set_smem_attr(const void* func, size_t bytes);

namespace {
inline size_t al256(size_t x) { return (x + 255) & ~(size_t)255; }

template <typename E, int DK, int DV>
gdn_status launch_job(const BwdParams& p, cudaStream_t s) {
    using J = BwdJob<E, DK, DV>;
    const size_t smem = sizeof(typename J::Smem);
    gdn_status st = set_smem_attr((const void*)bwd_job_kernel<E, DK, DV>, smem);
    if (st != GDN_OK) return st;
    bwd_job_kernel<E, DK, DV><<<dim3(p.num_seqs, p.Hv), NTB, smem, s>>>(p);
    return check_launch("bwd_job_kernel");
}

template <typename E, int DK>
gdn_status launch_dv(const BwdParams& p, cudaStream_t s) {
    switch (p.dv) {
        case 32: return launch_job<E, DK, 32>(p, s);
        case 64: return launch_job<E, DK, 64>(p, s);
        case 128: return launch_job<E, DK, 128>(p, s);
    }
    return fail(GDN_ERR_UNSUPPORTED_SHAPE, "backward: dv must be 32, 64 or 128");
}

template <typename E>
gdn_status launch_all(BwdParams p, cudaStream_t s) {
    const int rows = p.T * p.Hk;
    if (p.T > 0 && p.l2) {
        bwd_norms_kernel<E><<<(rows * 32 + 255) / 256, 256, 0, s>>>(
            static_cast<const E*>(p.q), static_cast<const E*>(p.k), p.ldq, p.ldk, p.T, p.Hk, p.dk,
            const_cast<float*>(p.rq), const_cast<float*>(p.rk));
        gdn_status st = check_launch("bwd_norms_kernel");
        if (st != GDN_OK) return st;
    }
    gdn_status st;
    switch (p.dk) {
        case 32: st = launch_dv<E, 32>(p, s); break;
        case 64: st = launch_dv<E, 64>(p, s); break;
        case 128: st = launch_dv<E, 128>(p, s); break;
        default: return fail(GDN_ERR_UNSUPPORTED_SHAPE, "backward: dk must be 32, 64 or 128");
    }
    if (st != GDN_OK) return st;
    if (p.T > 0 && p.l2) {
        bwd_l2_kernel<E><<<(2 * rows * 32 + 255) / 256, 256, 0, s>>>(
            static_cast<const E*>(p.q), static_cast<const E*>(p.k), p.ldq, p.ldk, p.T, p.Hk, p.dk, p.rq, p.rk,
            p.dq, p.dk_);
        st = check_launch("bwd_l2_kernel");
    }
    return st;
}
}  // namespace

size_t chunk_bwd_workspace_bytes(int T, int num_seqs, int Hk, int Hv, int dk, int dv) {
    const size_t state = (size_t)dk * dv * sizeof(float);
    return 2 * al256((size_t)T * Hk * sizeof(float)) +
           al256(((size_t)T / kSub + num_seqs + 1) * Hv * state) +
           al256((size_t)num_seqs * Hv * kSub * state);
}

gdn_status launch_chunk_bwd(const void* q, const void* k, const void* v, int64_t ldq, int64_t ldk, int64_t ldv,
                            gdn_dtype dtype, const float* g, const void* beta, const float* h0, const void* dout,
                            const float* dh_final, const int32_t* cu, int num_seqs, int T, int Hk, int Hv, int dk,
                            int dv, float scale, int l2, float* dq, float* dk_, float* dv_, float* dg, float* dbeta,
                            float* dh0, void* workspace, cudaStream_t s) {
    BwdParams p{};
    p.q = q; p.k = k; p.v = v; p.ldq = ldq; p.ldk = ldk; p.ldv = ldv;
    p.g = g; p.beta = beta; p.h0 = h0; p.dout = dout; p.dh_final = dh_final; p.cu = cu;
    p.num_seqs = num_seqs; p.T = T; p.Hk = Hk; p.Hv = Hv; p.dk = dk; p.dv = dv;
    p.scale = scale; p.l2 = l2;
    p.dq = dq; p.dk_ = dk_; p.dv_ = dv_; p.dg = dg; p.dbeta = dbeta; p.dh0 = dh0;
    unsigned char* w = static_cast<unsigned char*>(workspace);
    const size_t rbytes = al256((size_t)T * Hk * sizeof(float));
    const size_t state = (size_t)dk * dv * sizeof(float);
    p.rq = reinterpret_cast<float*>(w);
    p.rk = reinterpret_cast<float*>(w + rbytes);
    p.ckpt = reinterpret_cast<float*>(w + 2 * rbytes);
    p.scratch = reinterpret_cast<float*>(w + 2 * rbytes + al256(((size_t)T / kSub + num_seqs + 1) * Hv * state));
    // q/k gradients collect the value heads of a q/k head: start from zero
    if (T > 0) {
        if (cudaMemsetAsync(dq, 0, sizeof(float) * (size_t)T * Hk * dk, s) != cudaSuccess ||
            cudaMemsetAsync(dk_, 0, sizeof(float) * (size_t)T * Hk * dk, s) != cudaSuccess)
            return fail(GDN_ERR_CUDA, "backward: zeroing dq/dk failed");
    }
    if (dtype == GDN_BF16) return launch_all<__nv_bfloat16>(p, s);
    if (dtype == GDN_F32) return launch_all<float>(p, s);
    return fail(GDN_ERR_DTYPE, "backward: dtype must be bf16 or fp32");
}

}  // namespace gdn
