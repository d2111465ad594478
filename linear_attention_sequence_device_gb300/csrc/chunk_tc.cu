// bf16 chunk kernel for d_k = d_v = 128 on the 5th-generation tensor cores
// (tcgen05.mma, accumulators in tensor memory).
//
// One CTA (8 warps) runs one job: a token range of one value head with the
// full 128-column state, chunk after chunk (C = 64).  Every product is
// written transposed so that its M dimension is 128 (a head dimension):
//   Gram     [Q;K] [Q;K]^T             -> [128 x 128]  (Q K^T and K K^T blocks, norms on the diagonal)
//   W^T      K^T (T diag(beta e^G))^T  -> [128 x 64]
//   U^T      V^T (T diag(beta))^T      -> [128 x 64]
//   v_new^T  U^T - S^T W^T             -> [128 x 64]   (negated-A accumulate)
//   o^T      S^T Q~^T + v_new^T A^T    -> [128 x 64]   (Q~ = scale e^G Q)
//   dS^T     (v_new o e^{G_last-G})^T K -> [128 x 128]
// Operands sit in shared memory in the 128-byte-swizzled canonical layout;
// one tile serves as K-major operand of one product and MN-major operand of
// another.  The fp32 state S^T is held in registers (thread = value row,
// each warpgroup one half of the key columns) and copied to shared memory
// in bf16 as the A operand of the next chunk.  The Gram product is taken as
// [Q;K][Q;K]^T so that its diagonal gives the q/k L2 norms, which are then
// folded into scale factors (q and k are never rewritten normalised).  The
// 64x64 UT inverse runs in place with tf32 mma.sync block products.  Waits
// on the tensor core are bounded: on expiry the kernel counts a timeout,
// frees its tensor memory and returns.
#include "chunk_common.cuh"
#include "tc_util.cuh"

namespace gdn {

__device__ int g_gdn_timeouts;  // bounded waits that expired (read by gdn_device_timeouts)

namespace {

constexpr int NT = 256;
constexpr int LDF = 68;
constexpr uint32_t kSpin = 1u << 24;  // try_wait polls before a wait is declared stuck
typedef __nv_bfloat16 bf16;

struct SmemTC {
    bf16 QK[128 * 128];  // rows 0-63: Q (rescaled to scale e^G Q / |q| after the Gram), 64-127: K
    bf16 V[64 * 128];    // [token][value column]
    bf16 W[64 * 128];    // [token][key column]
    bf16 S[128 * 128];   // S^T [value column][key column], bf16 copy of the state
    bf16 Aqk[64 * 64];   // scale Q^ K^T o Gamma (lower incl. diagonal) [i][j]
    bf16 Tb[64 * 64];    // T diag(beta)
    bf16 Tbg[64 * 64];   // T diag(beta e^G / |k|)
    union {
        float LT[64 * LDF];      // L, then T = (I + L)^-1 in place
        struct {
            bf16 VN[128 * 64];   // v_new^T [value column][token]
            bf16 VNd[128 * 64];  // (v_new o e^{G_last - G} / |k|)^T
        } vn;
    } u;
    float g[64], beta[64], G[64], eG[64], eGl[64];
    float rn[128];       // 1/|q_i| (rows 0-63), 1/|k_j| (64-127); 1 without the L2-norm flag
    uint64_t mbar;
    uint32_t tmem_slot;
};

constexpr uint32_t ID_N64 = tc::idesc_bf16(128, 64, false, false, false);
constexpr uint32_t ID_N128 = tc::idesc_bf16(128, 128, false, false, false);
constexpr uint32_t ID_N64_AMN = tc::idesc_bf16(128, 64, true, false, false);
constexpr uint32_t ID_N64_NEG = tc::idesc_bf16(128, 64, false, false, true);
constexpr uint32_t ID_N128_BMN = tc::idesc_bf16(128, 128, false, true, false);

__device__ __forceinline__ uint4 pack8(const float* f) {
    uint4 r;
    __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&r);
#pragma unroll
    for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
    return r;
}

__global__ void __launch_bounds__(NT, 1) chunk_tc_kernel(const ChunkParams p, const int src) {
    extern __shared__ unsigned char smem_raw[];
    SmemTC& sm = *reinterpret_cast<SmemTC*>(smem_raw + ((1024 - (tc::smem_addr(smem_raw) & 1023)) & 1023));
    ChunkJob job;
    if (!make_job(p, src, job)) return;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int wg = warp >> 2;                // which half of the columns this thread handles
    const int row = (warp & 3) * 32 + lane;  // tensor-memory lane = row of every [128 x N] product
    const int hv = job.hv, hk = hv / (p.Hv / p.Hk);
    const bf16* __restrict__ q = static_cast<const bf16*>(p.q);
    const bf16* __restrict__ k = static_cast<const bf16*>(p.k);
    const bf16* __restrict__ v = static_cast<const bf16*>(p.v);
    const bf16* __restrict__ beta = static_cast<const bf16*>(p.beta);
    bf16* __restrict__ o = static_cast<bf16*>(p.o);
    const bool l2 = (p.flags & GDN_QK_L2NORM) != 0;

    if (tid == 0) tc::mbar_init(&sm.mbar, 1);
    if (warp == 0) tc::tmem_alloc(&sm.tmem_slot, 512);
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tmem = sm.tmem_slot;
    const uint32_t lb = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t T_GRAM = tmem, T_W = tmem + 128, T_U = tmem + 192, T_O = tmem + 256, T_DS = tmem + 320;
    const uint32_t aQK = tc::smem_addr(sm.QK), aK = aQK + 64 * 128, aV = tc::smem_addr(sm.V);
    const uint32_t aW = tc::smem_addr(sm.W), aS = tc::smem_addr(sm.S), aA = tc::smem_addr(sm.Aqk);
    const uint32_t aTb = tc::smem_addr(sm.Tb), aTbg = tc::smem_addr(sm.Tbg);
    const uint32_t aVN = tc::smem_addr(sm.u.vn.VN), aVNd = tc::smem_addr(sm.u.vn.VNd);
    uint32_t phase = 0;
    bool alive = true;

    // fp32 state: S^T[row][64 wg + c]
    float Sr[64];
#pragma unroll
    for (int c = 0; c < 64; ++c) {
        const int d = 64 * wg + c;
        float s0 = 0.f;
        if (job.identity_init) s0 = (d == job.col0 + row) ? 1.f : 0.f;
        else if (job.init) s0 = job.init[(int64_t)d * job.init_ld + row];
        Sr[c] = s0;
    }
#pragma unroll
    for (int c8 = 0; c8 < 8; ++c8)
        *reinterpret_cast<uint4*>(&sm.S[tc::sw128_chunk(128, row, 8 * wg + c8)]) = pack8(&Sr[8 * c8]);

    auto wait_mma = [&]() -> bool {
        const bool done = tc::mbar_wait(&sm.mbar, phase, kSpin);
        phase ^= 1u;
        const bool all = __syncthreads_and(done) != 0;
        if (!all && tid == 0) atomicAdd(&g_gdn_timeouts, 1);
        tc::fence_after();
        return all;
    };

    const int nch = (job.t1 - job.t0 + 63) / 64;
    for (int ch = 0; ch < nch && alive; ++ch) {
        const int tb = job.t0 + ch * 64;
        const int valid = min(64, job.t1 - tb);
        __syncthreads();
        // ---- load the chunk; rows past the segment end read as zero ----
        for (int e = tid; e < 64 * 16; e += NT) {
            const int r = e >> 4, c8 = e & 15;
            const int64_t t = tb + (r < valid ? r : 0);
            const int nb = r < valid ? 16 : 0;
            cp_async16(&sm.QK[tc::sw128_chunk(128, r, c8)], q + t * p.ldq + (int64_t)hk * 128 + c8 * 8, nb);
            cp_async16(&sm.QK[tc::sw128_chunk(128, 64 + r, c8)], k + t * p.ldk + (int64_t)hk * 128 + c8 * 8, nb);
            if (!job.value_zero)
                cp_async16(&sm.V[tc::sw128_chunk(64, r, c8)], v + t * p.ldv + (int64_t)hv * 128 + c8 * 8, nb);
        }
        cp_async_commit();
        if (tid < 64) {
            const int64_t t = tb + tid;
            sm.g[tid] = tid < valid ? __ldg(p.g + t * p.Hv + hv) : 0.f;
            sm.beta[tid] = tid < valid ? __bfloat162float(beta[t * p.Hv + hv]) : 0.f;
        }
        cp_async_wait_all();
        __syncthreads();
        if (warp == 0) gate_prefix_warp0(sm.g, sm.G, sm.eG, sm.eGl);
        tc::fence_async_smem();
        __syncthreads();

        // ---- Gram products: [Q;K] [Q;K]^T (the diagonal gives the L2 norms) ----
        if (tid == 0) {
            tc::fence_after();
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
                tc::mma(T_GRAM, tc::desc_k(aQK, 128, kk), tc::desc_k(aQK, 128, kk), ID_N128, kk > 0);
            tc::commit(&sm.mbar);
        }
        if (!(alive = wait_mma())) break;
        if (wg == 0) {  // 1 / sqrt(|x|^2 + 1e-6) from the Gram diagonal (x . x for row x)
            float dg[32];
            tc::ld32(T_GRAM + lb + (row & ~31), dg);
            float d = dg[0];
#pragma unroll
            for (int c = 1; c < 32; ++c) d = (c == lane) ? dg[c] : d;
            sm.rn[row] = l2 ? rsqrtf(d + 1e-6f) : 1.f;
        }
        __syncthreads();
        {
            float gv[32];
            tc::ld32(T_GRAM + lb + 64 + 32 * wg, gv);
            const int i = row & 63;
            const float Gi = sm.G[i];
            if (row < 64) {  // A = scale Q^ K^T o Gamma, lower triangle incl. diagonal
                const float fi = p.scale * sm.rn[i];
                float a[32];
#pragma unroll
                for (int c = 0; c < 32; ++c) {
                    const int j = 32 * wg + c;
                    a[c] = (j <= i) ? fi * sm.rn[64 + j] * gv[c] * __expf(Gi - sm.G[j]) : 0.f;
                }
#pragma unroll
                for (int c8 = 0; c8 < 4; ++c8)
                    *reinterpret_cast<uint4*>(&sm.Aqk[tc::sw128_chunk(64, i, 4 * wg + c8)]) = pack8(&a[8 * c8]);
            } else {         // L = beta_i K^ K^T o Gamma, strictly lower
                const float fi = sm.beta[i] * sm.rn[row];
                float* Lrow = sm.u.LT + i * LDF + 32 * wg;
#pragma unroll
                for (int c = 0; c < 32; c += 4) {
                    float4 l4;
                    float* lv = &l4.x;
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int j = 32 * wg + c + e;
                        lv[e] = (j < i) ? fi * sm.rn[64 + j] * gv[c + e] * __expf(Gi - sm.G[j]) : 0.f;
                    }
                    *reinterpret_cast<float4*>(Lrow + c) = l4;
                }
            }
        }
        tc::fence_before();
        __syncthreads();
        unit_lower_inverse64_inplace<LDF>(sm.u.LT, tid, [] { __syncthreads(); });
        // ---- T diag(beta), T diag(beta e^G / |k|) in bf16; Q <- scale e^G Q / |q| ----
        for (int e = tid; e < 64 * 8; e += NT) {
            const int i = e >> 3, c8 = e & 7;
            const float* trow = sm.u.LT + i * LDF + 8 * c8;
            float tbv[8], tbg[8];
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const int j = 8 * c8 + c;
                tbv[c] = trow[c] * sm.beta[j];
                tbg[c] = tbv[c] * sm.eG[j] * sm.rn[64 + j];
            }
            *reinterpret_cast<uint4*>(&sm.Tb[tc::sw128_chunk(64, i, c8)]) = pack8(tbv);
            *reinterpret_cast<uint4*>(&sm.Tbg[tc::sw128_chunk(64, i, c8)]) = pack8(tbg);
        }
        if (job.write_o) {
            for (int e = tid; e < 64 * 16; e += NT) {
                const int r = e >> 4, c8 = e & 15;
                uint4* ptr = reinterpret_cast<uint4*>(&sm.QK[tc::sw128_chunk(128, r, c8)]);
                uint4 raw = *ptr;
                __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&raw);
                const float f = p.scale * sm.eG[r] * sm.rn[r];
                float x[8];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float2 t2 = __bfloat1622float2(h[i]);
                    x[2 * i] = t2.x * f;
                    x[2 * i + 1] = t2.y * f;
                }
                *ptr = pack8(x);
            }
        }
        tc::fence_async_smem();
        __syncthreads();

        // ---- W^T = K^T Tbg^T, U^T = V^T Tb^T ----
        if (tid == 0) {
            tc::fence_after();
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                tc::mma(T_W, tc::desc_mn(aK, 128 * 128, kk), tc::desc_k(aTbg, 64, kk), ID_N64_AMN, kk > 0);
                if (!job.value_zero)
                    tc::mma(T_U, tc::desc_mn(aV, 64 * 128, kk), tc::desc_k(aTb, 64, kk), ID_N64_AMN, kk > 0);
            }
            tc::commit(&sm.mbar);
        }
        if (!(alive = wait_mma())) break;
        {  // W [token][key column] <- W^T rows (thread = key column)
            float wv[32];
            tc::ld32(T_W + lb + 32 * wg, wv);
            bf16* wb = sm.W + (row >> 6) * 64 * 64 + 32 * wg * 64 + (row & 7);
            const int dch = (row & 63) >> 3;
#pragma unroll
            for (int c = 0; c < 32; ++c) wb[64 * c + ((dch ^ (c & 7)) << 3)] = __float2bfloat16_rn(wv[c]);
        }
        tc::fence_before();
        tc::fence_async_smem();
        __syncthreads();

        // ---- v_new^T = U^T - S^T W^T ----
        if (tid == 0) {
            tc::fence_after();
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
                tc::mma(T_U, tc::desc_k(aS, 128, kk), tc::desc_k(aW, 64, kk), ID_N64_NEG,
                        (!job.value_zero) || kk > 0);
            tc::commit(&sm.mbar);
        }
        if (!(alive = wait_mma())) break;
        {
            float vv[32];
            tc::ld32(T_U + lb + 32 * wg, vv);
#pragma unroll
            for (int c8 = 0; c8 < 4; ++c8) {
                float d8[8];
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const int j = 32 * wg + 8 * c8 + c;
                    d8[c] = vv[8 * c8 + c] * sm.eGl[j] * sm.rn[64 + j];
                }
                *reinterpret_cast<uint4*>(&sm.u.vn.VN[tc::sw128_chunk(128, row, 4 * wg + c8)]) = pack8(&vv[8 * c8]);
                *reinterpret_cast<uint4*>(&sm.u.vn.VNd[tc::sw128_chunk(128, row, 4 * wg + c8)]) = pack8(d8);
            }
        }
        tc::fence_before();
        tc::fence_async_smem();
        __syncthreads();

        // ---- o^T = S^T Q~^T + v_new^T A^T ; dS^T = VNd K ----
        if (tid == 0) {
            tc::fence_after();
            if (job.write_o) {
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    tc::mma(T_O, tc::desc_k(aS, 128, kk), tc::desc_k(aQK, 128, kk), ID_N64, kk > 0);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    tc::mma(T_O, tc::desc_k(aVN, 128, kk), tc::desc_k(aA, 64, kk), ID_N64, 1);
            }
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                tc::mma(T_DS, tc::desc_k(aVNd, 128, kk), tc::desc_mn(aK, 128 * 128, kk), ID_N128_BMN, kk > 0);
            tc::commit(&sm.mbar);
        }
        if (!(alive = wait_mma())) break;
        if (job.write_o) {
            float ov[32];
            tc::ld32(T_O + lb + 32 * wg, ov);
            bf16* ob = o + ((int64_t)(tb + 32 * wg) * p.Hv + hv) * 128 + row;
            const int64_t ostride = (int64_t)p.Hv * 128;
#pragma unroll
            for (int c = 0; c < 32; ++c)
                if (32 * wg + c < valid) ob[c * ostride] = __float2bfloat16_rn(ov[c]);
        }
        {  // S <- e^{G_last} S + dS
            const float a = sm.eG[63];
            float ds[32];
            tc::ld32(T_DS + lb + 64 * wg, ds);
#pragma unroll
            for (int c = 0; c < 32; ++c) Sr[c] = fmaf(a, Sr[c], ds[c]);
            tc::ld32(T_DS + lb + 64 * wg + 32, ds);
#pragma unroll
            for (int c = 0; c < 32; ++c) Sr[32 + c] = fmaf(a, Sr[32 + c], ds[c]);
#pragma unroll
            for (int c8 = 0; c8 < 8; ++c8)
                *reinterpret_cast<uint4*>(&sm.S[tc::sw128_chunk(128, row, 8 * wg + c8)]) = pack8(&Sr[8 * c8]);
        }
        tc::fence_before();
    }
    if (alive && job.fin) {
#pragma unroll
        for (int c = 0; c < 64; ++c) job.fin[(int64_t)(64 * wg + c) * job.fin_ld + row] = Sr[c];
    }
    if (!alive) {
        // a stuck wait: give the tensor core a last bounded chance to drain
        tc::mbar_wait(&sm.mbar, phase ^ 1u, kSpin);
    }
    tc::fence_before();
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc(tmem, 512);
}

}  // namespace

gdn_status set_smem_attr(const void* func, size_t bytes);

bool chunk_tc_eligible(gdn_dtype dt, int dk, int dv) { return dt == GDN_BF16 && dk == 128 && dv == 128; }

gdn_status launch_chunk_tc(const ChunkParams& p, int src, dim3 grid, cudaStream_t s) {
    const size_t smem = sizeof(SmemTC) + 1024;
    gdn_status st = set_smem_attr((const void*)chunk_tc_kernel, smem);
    if (st != GDN_OK) return st;
    chunk_tc_kernel<<<grid, NT, smem, s>>>(p, src);
    return check_launch("chunk_tc_kernel");
}

}  // namespace gdn
