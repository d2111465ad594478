// fp32 chunk kernel: the chunked gated delta rule with every product on the
// FFMA pipe (fp32 inputs must meet a 1e-4 relative error bar, which TF32 or
// bf16 tensor-core operands cannot).  One CTA = one job (token range, value
// head, tile of 32 state columns); all operands live in shared memory.
#include "chunk_common.cuh"

namespace gdn {
namespace {

constexpr int NT = 256;
constexpr int CT = 32;       // state columns per CTA
constexpr int LDL = 65;      // row stride of the 64x64 fp32 tiles

template <int DK>
struct SmemF32 {
    float Q[64][DK + 1];
    float K[64][DK + 1];
    float W[64][DK + 1];
    float V[64][CT + 1];     // value tile, later v_new
    float U[64][CT + 1];
    float S[DK][CT + 1];     // state tile
    float L[64 * LDL];
    float Tm[64 * LDL];
    float A[64 * LDL];       // scale Q K^T o Gamma (incl. diagonal)
    float X[3 * 16 * 17];
    float g[64], beta[64], G[64], eG[64], eGl[64];
};

template <int DK>
__global__ void __launch_bounds__(NT) chunk_f32_kernel(const ChunkParams p, const int src) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    SmemF32<DK>& sm = *reinterpret_cast<SmemF32<DK>*>(smem_raw);
    ChunkJob job;
    if (!make_job(p, src, job)) return;
    const int tid = threadIdx.x;
    const int hv = job.hv, hk = hv / (p.Hv / p.Hk);
    const float* __restrict__ q = static_cast<const float*>(p.q);
    const float* __restrict__ k = static_cast<const float*>(p.k);
    const float* __restrict__ v = static_cast<const float*>(p.v);
    float* __restrict__ o = static_cast<float*>(p.o);
    const bool l2 = (p.flags & GDN_QK_L2NORM) != 0;

    // initial state
    for (int e = tid; e < DK * CT; e += NT) {
        const int i = e / CT, c = e % CT;
        float s0 = 0.f;
        if (job.identity_init) s0 = (i == job.col0 + c) ? 1.f : 0.f;
        else if (job.init) s0 = job.init[(int64_t)i * job.init_ld + c];
        sm.S[i][c] = s0;
    }

    const int nch = (job.t1 - job.t0 + 63) / 64;
    for (int ch = 0; ch < nch; ++ch) {
        const int tb = job.t0 + ch * 64;
        const int valid = min(64, job.t1 - tb);
        __syncthreads();
        // ---- load the chunk (rows past the end are zero, beta = g = 0) ----
        for (int e = tid; e < 64 * DK; e += NT) {
            const int r = e / DK, d = e % DK;
            const bool ok = r < valid;
            const int64_t t = tb + r;
            sm.Q[r][d] = ok ? q[t * p.ldq + (int64_t)hk * p.hsq + d] : 0.f;
            sm.K[r][d] = ok ? k[t * p.ldk + (int64_t)hk * p.hsk + d] : 0.f;
        }
        for (int e = tid; e < 64 * CT; e += NT) {
            const int r = e / CT, c = e % CT;
            const int64_t t = tb + r;
            sm.V[r][c] = (r < valid && !job.value_zero)
                             ? v[t * p.ldv + (int64_t)hv * p.hsv + job.col0 + c] : 0.f;
        }
        if (tid < 64) {
            const int64_t t = tb + tid;
            float gv = 0.f, bv = 0.f;
            if (tid < valid) gate_beta<float>(p, t, hv, gv, bv);
            sm.g[tid] = gv;
            sm.beta[tid] = bv;
        }
        __syncthreads();
        if (l2) {  // q, k <- x * rsqrt(|x|^2 + 1e-6), one warp per row
            const int w = tid >> 5, lane = tid & 31;
            for (int r = w; r < 128; r += NT / 32) {
                float* row = r < 64 ? sm.Q[r] : sm.K[r - 64];
                float ss = 0.f;
                for (int d = lane; d < DK; d += 32) ss = fmaf(row[d], row[d], ss);
#pragma unroll
                for (int off = 16; off; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
                const float rn = rsqrtf(ss + 1e-6f);
                for (int d = lane; d < DK; d += 32) row[d] *= rn;
            }
        }
        if (tid < 32) gate_prefix_warp0(sm.g, sm.G, sm.eG, sm.eGl);
        __syncthreads();
        // ---- L (strict lower) and A = scale Q K^T o Gamma (lower incl.) ----
        for (int e = tid; e < 64 * 64; e += NT) {
            const int i = e >> 6, j = e & 63;
            float kk = 0.f, qk = 0.f;
            if (i >= j) {
                for (int d = 0; d < DK; ++d) {
                    kk = fmaf(sm.K[i][d], sm.K[j][d], kk);
                    qk = fmaf(sm.Q[i][d], sm.K[j][d], qk);
                }
            }
            const float gam = (i >= j) ? expf(sm.G[i] - sm.G[j]) : 0.f;
            sm.L[i * LDL + j] = (i > j) ? sm.beta[i] * kk * gam : 0.f;
            sm.A[i * LDL + j] = p.scale * qk * gam;
        }
        __syncthreads();
        unit_lower_inverse64<NT, LDL>(sm.L, sm.Tm, sm.X);
        // ---- W = T diag(beta e^G) K ; U = T diag(beta) V ----
        for (int e = tid; e < 64 * DK; e += NT) {
            const int i = e / DK, d = e % DK;
            float acc = 0.f;
            for (int j = 0; j <= i; ++j)
                acc = fmaf(sm.Tm[i * LDL + j] * sm.beta[j] * sm.eG[j], sm.K[j][d], acc);
            sm.W[i][d] = acc;
        }
        for (int e = tid; e < 64 * CT; e += NT) {
            const int i = e / CT, c = e % CT;
            float acc = 0.f;
            for (int j = 0; j <= i; ++j) acc = fmaf(sm.Tm[i * LDL + j] * sm.beta[j], sm.V[j][c], acc);
            sm.U[i][c] = acc;
        }
        __syncthreads();
        // ---- v_new = U - W S  (into V) ----
        for (int e = tid; e < 64 * CT; e += NT) {
            const int i = e / CT, c = e % CT;
            float acc = sm.U[i][c];
            for (int d = 0; d < DK; ++d) acc = fmaf(-sm.W[i][d], sm.S[d][c], acc);
            sm.V[i][c] = acc;
        }
        __syncthreads();
        // ---- o = scale e^G (Q S) + A v_new ----
        if (job.write_o) {
            for (int e = tid; e < 64 * CT; e += NT) {
                const int i = e / CT, c = e % CT;
                if (i >= valid) continue;
                float qs = 0.f;
                for (int d = 0; d < DK; ++d) qs = fmaf(sm.Q[i][d], sm.S[d][c], qs);
                float acc = p.scale * sm.eG[i] * qs;
                for (int j = 0; j <= i; ++j) acc = fmaf(sm.A[i * LDL + j], sm.V[j][c], acc);
                o[(int64_t)(tb + i) * p.ldo + (int64_t)hv * p.hso + job.col0 + c] = acc;
            }
        }
        __syncthreads();
        // ---- S <- e^{G_last} S + (K o e^{G_last - G})^T v_new ----
        const float eGlast = sm.eG[63];
        for (int e = tid; e < DK * CT; e += NT) {
            const int d = e / CT, c = e % CT;
            float acc = eGlast * sm.S[d][c];
            for (int j = 0; j < 64; ++j) acc = fmaf(sm.K[j][d] * sm.eGl[j], sm.V[j][c], acc);
            sm.S[d][c] = acc;
        }
    }
    __syncthreads();
    if (job.fin) {
        for (int e = tid; e < DK * CT; e += NT) {
            const int i = e / CT, c = e % CT;
            job.fin[(int64_t)i * job.fin_ld + c] = sm.S[i][c];
        }
    }
}

}  // namespace

gdn_status set_smem_attr(const void* func, size_t bytes);

namespace {
template <int DK>
gdn_status launch_dk(const ChunkParams& p, int src, dim3 grid, cudaStream_t s) {
    const size_t smem = sizeof(SmemF32<DK>);
    gdn_status st = set_smem_attr((const void*)chunk_f32_kernel<DK>, smem);
    if (st != GDN_OK) return st;
    chunk_f32_kernel<DK><<<grid, NT, smem, s>>>(p, src);
    return check_launch("chunk_f32_kernel");
}

}  // namespace

gdn_status launch_chunk_f32(const ChunkParams& p, int src, dim3 grid, cudaStream_t s) {
    switch (p.dk) {
        case 32: return launch_dk<32>(p, src, grid, s);
        case 64: return launch_dk<64>(p, src, grid, s);
        case 128: return launch_dk<128>(p, src, grid, s);
    }
    return fail(GDN_ERR_UNSUPPORTED_SHAPE, "dk=%d not in {32,64,128}", p.dk);
}

}  // namespace gdn
