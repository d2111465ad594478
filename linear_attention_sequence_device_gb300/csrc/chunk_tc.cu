// bf16 chunk kernel for d_k = d_v = 128 on the 5th-generation tensor cores
// (tcgen05.mma, accumulators in tensor memory).
//
// One CTA runs one job: a token range of one value head with the full
// 128-column state, chunk after chunk (C = 64).  Every product is written
// transposed so that its M dimension is 128 (a head dimension):
//   Gram     [Q;K] [Q;K]^T              -> [128 x 128] (Q K^T and K K^T blocks, norms on the diagonal)
//   W^T      K^T (T diag(beta e^G/|k|))^T -> [128 x 64]
//   U^T      V^T (T diag(beta))^T        -> [128 x 64]
//   v_new^T  U^T - S^T W^T               -> [128 x 64]   (negated-A accumulate)
//   o^T      S^T Q~^T + v_new^T A^T      -> [128 x 64]   (Q~ = scale e^G Q / |q|)
//   dS^T     (v_new o e^{G_last-G}/|k|)^T K -> [128 x 128]
// Operands sit in shared memory in the 128-byte-swizzled canonical layout;
// one tile serves as K-major operand of one product and MN-major operand of
// another.
//
// Two roles of two warpgroups each work on different chunks at once (the
// two warpgroups of a role split the columns of every elementwise step):
//   producer (warps 0-7): everything that does not depend on the state --
//     loads, the Gram product, the L2 norms (from the Gram diagonal, folded
//     into scale factors), A and L, the in-place UT inverse (tf32 mma.sync
//     block products), W and U -- for chunk c+1 while
//   consumer (warps 8-15) runs the state chain of chunk c: v_new, then o and
//     dS, then S <- e^{G_last} S + dS with the fp32 state in registers
//     (thread = value row, half the key columns) and a bf16 copy in shared memory as the A operand.
// Q/K, A, the per-chunk scale factors and U (in tensor memory) are double
// buffered ("slots"); W is single buffered with its own release barrier.
// Every wait is bounded: on expiry the kernel counts a timeout, both groups
// leave their loops, and the tensor memory is freed.
#include <cuda.h>
#include <string.h>

#include "chunk_common.cuh"
#include "tc_util.cuh"

namespace gdn {

__device__ int g_gdn_timeouts;  // bounded waits that expired (read by gdn_device_timeouts)

namespace {

constexpr int NT = 512;
constexpr int GS = 256;  // threads per role (two warpgroups)
constexpr int LDF = 68;
constexpr uint32_t kSpin = 1u << 20;  // try_wait polls before a wait is declared stuck
constexpr int BAR_P = 1, BAR_S = 2;   // named barriers of the two roles
constexpr int BAR_PA = 3;             // producer warps 0-3 (the UT inverse)
typedef __nv_bfloat16 bf16;

struct TmaMaps {
    CUtensorMap q, k, v;  // [T rows x heads*128 columns] bf16 views, 64x64 boxes, 128-byte swizzle
};

struct SlotSmall {
    float fac[64];  // e^{G_last - G_j} / |k_j|: token factor of dS
    float eglast;   // e^{G_last}
    int tb, valid;  // first token and valid rows of the chunk
    int pad;
};

struct SmemWS {
    bf16 QK[2][128 * 128];  // per slot: rows 0-63 Q (then Q~), rows 64-127 K
    bf16 Aqk[2][64 * 64];   // per slot: scale Q^ K^T o Gamma, lower incl. diagonal
    bf16 W[64 * 128];       // [token][key column]
    bf16 V[64 * 128];       // [token][value column]
    bf16 S[128 * 128];      // S^T [value column][key column] (bf16 copy of the state)
    bf16 VN[128 * 64];      // v_new^T [value column][token]
    bf16 VNd[128 * 64];     // v_new^T scaled by the dS token factor
    bf16 Tb[64 * 64];       // T diag(beta)
    bf16 Tbg[64 * 64];      // T diag(beta e^G / |k|)
    float LT[64 * LDF];     // L, then T = (I + L)^-1 in place
    SlotSmall slot[2];
    float g[64], beta[64], G[64], eG[64], eGl[64];
    float rn[128];          // 1/|q_i| (0-63), 1/|k_j| (64-127); 1 without the L2-norm flag
    // per-chunk factors; e^{G_i - G_j} = e^{G_i - G_r} e^{G_r - G_j} with G_r = G_31
    float colf[64];         // e^{G_r - G_j} / |k_j|
    float rowA[64];         // scale e^{G_i - G_r} / |q_i|
    float rowL[64];         // beta_i e^{G_i - G_r} / |k_i|
    float fbg[64];          // beta_j e^{G_j} / |k_j|
    float qf[64];           // scale e^{G_i} / |q_i|
    int factored;           // the split exponentials stay well inside fp32 range
    uint64_t mbar_p, mbar_s;  // tensor-core completion, producer / consumer
    uint64_t full[2], empty[2], wfree;
    uint64_t ld_qk[2], ld_v;   // TMA arrivals (transaction bytes)
    uint32_t tmem_slot;
    int lpt_len[kMaxLptItems];
    int lpt_pick;
};

constexpr uint32_t ID_N64 = tc::idesc_bf16(128, 64, false, false, false);
constexpr uint32_t ID_N128 = tc::idesc_bf16(128, 128, false, false, false);
constexpr uint32_t ID_N64_AMN = tc::idesc_bf16(128, 64, true, false, false);
constexpr uint32_t ID_N64_NEG = tc::idesc_bf16(128, 64, false, false, true);
constexpr uint32_t ID_N128_BMN = tc::idesc_bf16(128, 128, false, true, false);

// One warp: the chunk's gate prefix from per-token values held by lanes
// (lane l holds g of tokens 2l and 2l+1; beta likewise), written to shared
// memory with e^G, e^{G_last - G}, beta, and whether split exponentials
// around G_31 stay within fp32 range.
template <class Sm>
__device__ __forceinline__ void gate_prefix_fast(Sm& sm, float g0, float g1, float b0, float b1) {
    const int lane = threadIdx.x & 31;
    float s = g0 + g1;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const float t = __shfl_up_sync(0xffffffffu, s, off);
        if (lane >= off) s += t;
    }
    const float G1 = s, G0 = s - g1;
    const float Gl = __shfl_sync(0xffffffffu, s, 31);
    const float Gr = __shfl_sync(0xffffffffu, s, 15);  // G_31 = inclusive sum through token 31
    sm.G[2 * lane] = G0;
    sm.G[2 * lane + 1] = G1;
    sm.eG[2 * lane] = __expf(G0);
    sm.eG[2 * lane + 1] = __expf(G1);
    sm.eGl[2 * lane] = __expf(Gl - G0);
    sm.eGl[2 * lane + 1] = __expf(Gl - G1);
    sm.beta[2 * lane] = b0;
    sm.beta[2 * lane + 1] = b1;
    float dev = fmaxf(fabsf(G0 - Gr), fabsf(G1 - Gr));
#pragma unroll
    for (int off = 16; off; off >>= 1) dev = fmaxf(dev, __shfl_xor_sync(0xffffffffu, dev, off));
    if (lane == 0) sm.factored = dev < 60.f;
}

__device__ __forceinline__ uint4 pack8(const float* f) {
    uint4 r;
    __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&r);
#pragma unroll
    for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
    return r;
}

__global__ void __launch_bounds__(NT, 1) chunk_tc_kernel(const ChunkParams p, const int src,
                                                        const __grid_constant__ TmaMaps maps) {
    extern __shared__ unsigned char smem_raw[];
    SmemWS& sm = *reinterpret_cast<SmemWS*>(smem_raw + ((1024 - (tc::smem_addr(smem_raw) & 1023)) & 1023));
    ChunkJob job;
    int bx, by, bz;
    lpt_block<NT>(p, src, sm.lpt_len, &sm.lpt_pick, bx, by, bz);
    if (!make_job(p, src, job, bx, by, bz)) return;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const bool producer = warp < 8;
    const int gt = tid & (GS - 1);  // thread index in its role
    const int row = gt & 127;       // tensor-memory lane = row of every [128 x N] product
    const int half = gt >> 7;       // which half of the columns this thread handles
    const uint32_t lb = (uint32_t)((warp & 3) * 32) << 16;
    const int hv = job.hv, hk = hv / (p.Hv / p.Hk);

    if (tid == 0) {
        tc::mbar_init(&sm.mbar_p, 1);
        tc::mbar_init(&sm.mbar_s, 1);
        tc::mbar_init(&sm.full[0], 1);
        tc::mbar_init(&sm.full[1], 1);
        tc::mbar_init(&sm.empty[0], 1);
        tc::mbar_init(&sm.empty[1], 1);
        tc::mbar_init(&sm.wfree, 1);
        tc::mbar_init(&sm.ld_qk[0], 1);
        tc::mbar_init(&sm.ld_qk[1], 1);
        tc::mbar_init(&sm.ld_v, 1);
    }
    if (warp == 0) tc::tmem_alloc(&sm.tmem_slot, 512);
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tmem = sm.tmem_slot;
    const uint32_t T_GRAM = tmem, T_W = tmem + 128, T_O = tmem + 320, T_DS = tmem + 384;
    // per-slot values are picked with selects (a runtime-indexed array would live in local memory)
    const uint32_t T_U0 = tmem + 192, T_U1 = tmem + 256;
    const uint32_t aQK0 = tc::smem_addr(sm.QK[0]), aQK1 = tc::smem_addr(sm.QK[1]);
    const uint32_t aA0 = tc::smem_addr(sm.Aqk[0]), aA1 = tc::smem_addr(sm.Aqk[1]);
    const uint32_t aW = tc::smem_addr(sm.W), aV = tc::smem_addr(sm.V), aS = tc::smem_addr(sm.S);
    const uint32_t aVN = tc::smem_addr(sm.VN), aVNd = tc::smem_addr(sm.VNd);
    const uint32_t aTb = tc::smem_addr(sm.Tb), aTbg = tc::smem_addr(sm.Tbg);
    const int nch = (job.t1 - job.t0 + 63) / 64;
    bool ok = true;
    // base descriptors; a K step adds a constant to the start-address field
    const uint64_t dQK0 = tc::desc(aQK0, 16, 1024), dQK1 = tc::desc(aQK1, 16, 1024);
    const uint64_t dKmn0 = tc::desc(aQK0 + 64 * 128, 128 * 128, 1024), dKmn1 = tc::desc(aQK1 + 64 * 128, 128 * 128, 1024);
    const uint64_t dA0 = tc::desc(aA0, 16, 1024), dA1 = tc::desc(aA1, 16, 1024);
    const uint64_t dW = tc::desc(aW, 16, 1024), dVmn = tc::desc(aV, 64 * 128, 1024), dS = tc::desc(aS, 16, 1024);
    const uint64_t dVN = tc::desc(aVN, 16, 1024), dVNd = tc::desc(aVNd, 16, 1024);
    const uint64_t dTb = tc::desc(aTb, 16, 1024), dTbg = tc::desc(aTbg, 16, 1024);

    if (producer) {
        // ====================== producer warpgroup ======================
        const bf16* __restrict__ beta = static_cast<const bf16*>(p.beta);
        const bool l2 = (p.flags & GDN_QK_L2NORM) != 0;
        uint32_t ph = 0;
        auto wait_mma = [&]() -> bool {
            const bool done = tc::mbar_wait(&sm.mbar_p, ph, kSpin);
            ph ^= 1u;
            const bool all = tc::bar_and(BAR_P, GS, done);
            tc::fence_after();
            return all;
        };
        // TMA loads: Q/K of chunk cc into its slot (four 64x64 boxes, 128-byte
        // swizzle = the operand layout), V into the single V tile (two boxes);
        // g and beta into registers, stored to shared memory at the chunk's start
        float g_next0 = 0.f, g_next1 = 0.f, b_next0 = 0.f, b_next1 = 0.f;
        auto issue_qk = [&](int cc) {
            const int tbn = job.t0 + 64 * cc;
            const int vn = min(64, job.t1 - tbn);
            if (gt == 0) {
                bf16* QKn = sm.QK[cc & 1];
                uint64_t* bar = &sm.ld_qk[cc & 1];
                tc::mbar_expect_tx(bar, 4 * 64 * 64 * 2);
                tc::tma_load_2d(QKn, &maps.q, hk * 128, tbn, bar);
                tc::tma_load_2d(QKn + 128 * 64, &maps.q, hk * 128 + 64, tbn, bar);
                tc::tma_load_2d(QKn + 64 * 64, &maps.k, hk * 128, tbn, bar);
                tc::tma_load_2d(QKn + 128 * 64 + 64 * 64, &maps.k, hk * 128 + 64, tbn, bar);
            }
            if (warp == 0) {  // lane l: tokens 2l, 2l+1
                const int r0 = 2 * lane, r1 = 2 * lane + 1;
                const int64_t t0 = tbn + r0, t1 = tbn + r1;
                g_next0 = r0 < vn ? __ldg(p.g + t0 * p.Hv + hv) : 0.f;
                g_next1 = r1 < vn ? __ldg(p.g + t1 * p.Hv + hv) : 0.f;
                b_next0 = r0 < vn ? __bfloat162float(beta[t0 * p.Hv + hv]) : 0.f;
                b_next1 = r1 < vn ? __bfloat162float(beta[t1 * p.Hv + hv]) : 0.f;
            }
        };
        auto issue_v = [&](int cc) {
            if (gt == 0 && !job.value_zero) {
                const int tbn = job.t0 + 64 * cc;
                tc::mbar_expect_tx(&sm.ld_v, 2 * 64 * 64 * 2);
                tc::tma_load_2d(sm.V, &maps.v, hv * 128, tbn, &sm.ld_v);
                tc::tma_load_2d(sm.V + 64 * 64, &maps.v, hv * 128 + 64, tbn, &sm.ld_v);
            }
        };
        auto wait_bar = [&](uint64_t* bar, uint32_t parity) -> bool {
            const bool all = tc::bar_and(BAR_P, GS, tc::mbar_wait(bar, parity, kSpin));
            tc::fence_after();
            return all;
        };
        // the Gram product [Q;K][Q;K]^T of the chunk in slot ss (diagonal: the L2 norms)
        auto issue_gram = [&](int ss) {
            if (gt == 0) {
                tc::fence_after();
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    tc::mma(T_GRAM, (ss ? dQK1 : dQK0) + tc::koff(128, kk), (ss ? dQK1 : dQK0) + tc::koff(128, kk),
                            ID_N128, kk > 0);
                tc::commit(&sm.mbar_p);
            }
        };
        if (nch > 0) {
            issue_qk(0);
            issue_v(0);
            if ((ok = wait_bar(&sm.ld_qk[0], 0))) issue_gram(0);
            if (warp == 0) gate_prefix_fast(sm, g_next0, g_next1, b_next0, b_next1);
        }
        for (int c = 0; c < nch && ok; ++c) {
            const int s = c & 1;
            const int tb = job.t0 + 64 * c;
            const int valid = min(64, job.t1 - tb);
            bf16* QKs = sm.QK[s];
            // the gate prefix of this chunk was formed at the end of the previous one
            if (!(ok = wait_mma())) break;  // the Gram product of this chunk
            if (half == 0) {  // 1 / sqrt(|x|^2 + 1e-6) from the diagonal
                float dg[32];
                tc::ld32(T_GRAM + lb + (row & ~31), dg);
                float d = dg[0];
#pragma unroll
                for (int c2 = 1; c2 < 32; ++c2) d = (c2 == lane) ? dg[c2] : d;
                const float r = l2 ? rsqrtf(d + 1e-6f) : 1.f;
                sm.rn[row] = r;
                const int i = row & 63;
                const float Gi = sm.G[i], Gr = sm.G[31];
                if (row < 64) {
                    sm.rowA[i] = p.scale * r * __expf(Gi - Gr);
                    sm.qf[i] = p.scale * sm.eG[i] * r;
                } else {
                    sm.colf[i] = r * __expf(Gr - Gi);
                    sm.rowL[i] = sm.beta[i] * r * __expf(Gi - Gr);
                    sm.fbg[i] = sm.beta[i] * sm.eG[i] * r;
                }
            }
            tc::bar_sync(BAR_P, GS);
            {  // A (rows 0-63) and L (rows 64-127) from the Q K^T / K K^T blocks
                const int i = row & 63;
                float gv[32];
                tc::ld32(T_GRAM + lb + 64 + 32 * half, gv);
                float a[32];
                if (sm.factored) {
                    const float fi = row < 64 ? sm.rowA[i] : sm.rowL[i];
                    const int lim = row < 64 ? i : i - 1;  // A keeps the diagonal, L does not
                    const float4* cf = reinterpret_cast<const float4*>(sm.colf + 32 * half);
#pragma unroll
                    for (int c4 = 0; c4 < 8; ++c4) {
                        const float4 f4 = cf[c4];
                        const float fc[4] = {f4.x, f4.y, f4.z, f4.w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int c2 = 4 * c4 + e;
                            a[c2] = (32 * half + c2 <= lim) ? fi * (fc[e] * gv[c2]) : 0.f;
                        }
                    }
                } else {  // wide gate range: one exponential per element
                    const float Gi = sm.G[i];
                    const float fi = row < 64 ? p.scale * sm.rn[i] : sm.beta[i] * sm.rn[row];
                    const int lim = row < 64 ? i : i - 1;
#pragma unroll
                    for (int c2 = 0; c2 < 32; ++c2) {
                        const int j = 32 * half + c2;
                        a[c2] = (j <= lim) ? fi * sm.rn[64 + j] * gv[c2] * __expf(Gi - sm.G[j]) : 0.f;
                    }
                }
                if (row < 64) {
#pragma unroll
                    for (int c8 = 0; c8 < 4; ++c8)
                        *reinterpret_cast<uint4*>(&sm.Aqk[s][tc::sw128_chunk(64, i, 4 * half + c8)]) = pack8(&a[8 * c8]);
                } else {
                    float4* Lrow = reinterpret_cast<float4*>(sm.LT + i * LDF + 32 * half);
#pragma unroll
                    for (int c4 = 0; c4 < 8; ++c4)
                        Lrow[c4] = make_float4(a[4 * c4], a[4 * c4 + 1], a[4 * c4 + 2], a[4 * c4 + 3]);
                }
            }
            tc::fence_before();
            tc::bar_sync(BAR_P, GS);
            // the UT inverse on warps 0-3; warps 4-7 rescale Q meanwhile
            if (gt < 128) {
                unit_lower_inverse64_rec<LDF>(sm.LT, gt, [] { tc::bar_sync(BAR_PA, 128); });
            } else if (job.write_o) {
                for (int e = gt - 128; e < 64 * 16; e += 128) {
                    const int r = e >> 4, c8 = e & 15;
                    uint4* ptr = reinterpret_cast<uint4*>(&QKs[tc::sw128_chunk(128, r, c8)]);
                    uint4 raw = *ptr;
                    __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&raw);
                    const float f = sm.qf[r];
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
            tc::bar_sync(BAR_P, GS);
            // T diag(beta), T diag(beta e^G / |k|); slot factors
            for (int e = gt; e < 64 * 8; e += GS) {
                const int i = e >> 3, c8 = e & 7;
                const float4* trow = reinterpret_cast<const float4*>(sm.LT + i * LDF + 8 * c8);
                const float4* bj = reinterpret_cast<const float4*>(sm.beta + 8 * c8);
                const float4* fj = reinterpret_cast<const float4*>(sm.fbg + 8 * c8);
                float tbv[8], tbg[8];
#pragma unroll
                for (int h2 = 0; h2 < 2; ++h2) {
                    const float4 t4 = trow[h2], b4 = bj[h2], f4 = fj[h2];
                    tbv[4 * h2] = t4.x * b4.x; tbv[4 * h2 + 1] = t4.y * b4.y;
                    tbv[4 * h2 + 2] = t4.z * b4.z; tbv[4 * h2 + 3] = t4.w * b4.w;
                    tbg[4 * h2] = t4.x * f4.x; tbg[4 * h2 + 1] = t4.y * f4.y;
                    tbg[4 * h2 + 2] = t4.z * f4.z; tbg[4 * h2 + 3] = t4.w * f4.w;
                }
                *reinterpret_cast<uint4*>(&sm.Tb[tc::sw128_chunk(64, i, c8)]) = pack8(tbv);
                *reinterpret_cast<uint4*>(&sm.Tbg[tc::sw128_chunk(64, i, c8)]) = pack8(tbg);
            }
            if (gt < 64) sm.slot[s].fac[gt] = sm.eGl[gt] * sm.rn[64 + gt];
            if (gt == 0) {
                sm.slot[s].eglast = sm.eG[63];
                sm.slot[s].tb = tb;
                sm.slot[s].valid = valid;
            }
            tc::fence_async_smem();
            tc::bar_sync(BAR_P, GS);
            // W^T = K^T Tbg^T, U^T = V^T Tb^T (V of this chunk must have landed)
            if (!job.value_zero && !(ok = wait_bar(&sm.ld_v, c & 1))) break;
            if (gt == 0) {
                tc::fence_after();
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    tc::mma(T_W, (s ? dKmn1 : dKmn0) + tc::mnoff(kk), dTbg + tc::koff(64, kk), ID_N64_AMN, kk > 0);
                    if (!job.value_zero)
                        tc::mma((s ? T_U1 : T_U0), dVmn + tc::mnoff(kk), dTb + tc::koff(64, kk), ID_N64_AMN, kk > 0);
                }
                tc::commit(&sm.mbar_p);
            }
            // prefetch chunk c+1 while W and U form: its Q/K slot once the
            // consumer has released it (chunk c-1); V once U no longer reads it
            if (c + 1 < nch) {
                if (c >= 1 && !(ok = wait_bar(&sm.empty[s ^ 1], ((c - 1) >> 1) & 1))) break;
                issue_qk(c + 1);
            }
            if (!(ok = wait_mma())) break;
            if (c + 1 < nch) issue_v(c + 1);
            // W goes to shared memory once the consumer's v_new of chunk c-1 is done with it
            if (c >= 1 && !(ok = wait_bar(&sm.wfree, (c - 1) & 1))) break;
            {
                float wv[32];
                const int dch = (row & 63) >> 3;
                tc::ld32(T_W + lb + 32 * half, wv);
                bf16* wb = sm.W + (row >> 6) * 64 * 64 + 32 * half * 64 + (row & 7);
#pragma unroll
                for (int c2 = 0; c2 < 32; ++c2) wb[64 * c2 + ((dch ^ (c2 & 7)) << 3)] = __float2bfloat16_rn(wv[c2]);
            }
            tc::fence_async_smem();
            tc::fence_before();
            tc::bar_sync(BAR_P, GS);
            if (gt == 0) tc::mbar_arrive(&sm.full[s]);
            // the next chunk's Gram product starts as soon as its Q/K are in,
            // and its gate prefix is formed meanwhile (this chunk no longer reads G)
            if (c + 1 < nch) {
                if (!(ok = wait_bar(&sm.ld_qk[s ^ 1], ((c + 1) >> 1) & 1))) break;
                issue_gram(s ^ 1);
                if (warp == 0) gate_prefix_fast(sm, g_next0, g_next1, b_next0, b_next1);
            }
        }
    } else {
        // ====================== consumer warpgroup ======================
        bf16* __restrict__ o = static_cast<bf16*>(p.o);
        uint32_t ph = 0;
        auto wait_mma = [&]() -> bool {
            const bool done = tc::mbar_wait(&sm.mbar_s, ph, kSpin);
            ph ^= 1u;
            const bool all = tc::bar_and(BAR_S, GS, done);
            tc::fence_after();
            return all;
        };
        // state S^T row `row` (value column), key columns [64 half, 64 half + 64)
        float Sr[64];
#pragma unroll
        for (int c2 = 0; c2 < 64; ++c2) {
            const int d = 64 * half + c2;
            float s0 = 0.f;
            if (job.identity_init) s0 = (d == job.col0 + row) ? 1.f : 0.f;
            else if (job.init) s0 = job.init[(int64_t)d * job.init_ld + row];
            Sr[c2] = s0;
        }
#pragma unroll
        for (int c8 = 0; c8 < 8; ++c8)
            *reinterpret_cast<uint4*>(&sm.S[tc::sw128_chunk(128, row, 8 * half + c8)]) = pack8(&Sr[8 * c8]);
        tc::fence_async_smem();
        tc::bar_sync(BAR_S, GS);
        const int64_t ostride = (int64_t)p.Hv * 128;
        auto store_o = [&](int otb, int ovalid) {
            float ov[32];
            tc::ld32(T_O + lb + 32 * half, ov);
            bf16* ob = o + ((int64_t)(otb + 32 * half) * p.Hv + hv) * 128 + row;
#pragma unroll
            for (int c2 = 0; c2 < 32; ++c2)
                if (32 * half + c2 < ovalid) ob[c2 * ostride] = __float2bfloat16_rn(ov[c2]);
        };
        int o_tb = 0, o_valid = 0;
        bool o_pending = false;
        for (int c = 0; c < nch; ++c) {
            const int s = c & 1;
            if (!(ok = tc::bar_and(BAR_S, GS, tc::mbar_wait(&sm.full[s], (c >> 1) & 1, kSpin)))) break;
            tc::fence_after();
            // v_new^T = U^T - S^T W^T
            if (gt == 0) {
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    tc::mma((s ? T_U1 : T_U0), dS + tc::koff(128, kk), dW + tc::koff(64, kk), ID_N64_NEG,
                            (!job.value_zero) || kk > 0);
                tc::commit(&sm.mbar_s);
            }
            if (o_pending) store_o(o_tb, o_valid);  // previous chunk's output, while the MMA runs
            if (!(ok = wait_mma())) break;
            if (gt == 0) tc::mbar_arrive(&sm.wfree);
            {
                const float* fac = sm.slot[s].fac;
                float vv[32];
                tc::ld32((s ? T_U1 : T_U0) + lb + 32 * half, vv);
#pragma unroll
                for (int c8 = 0; c8 < 4; ++c8) {
                    float d8[8];
#pragma unroll
                    for (int c2 = 0; c2 < 8; ++c2) d8[c2] = vv[8 * c8 + c2] * fac[32 * half + 8 * c8 + c2];
                    *reinterpret_cast<uint4*>(&sm.VN[tc::sw128_chunk(128, row, 4 * half + c8)]) = pack8(&vv[8 * c8]);
                    *reinterpret_cast<uint4*>(&sm.VNd[tc::sw128_chunk(128, row, 4 * half + c8)]) = pack8(d8);
                }
            }
            tc::fence_async_smem();
            tc::fence_before();
            tc::bar_sync(BAR_S, GS);
            // o^T = S^T Q~^T + v_new^T A^T ; dS^T = VNd K
            if (gt == 0) {
                tc::fence_after();
                if (job.write_o) {
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)
                        tc::mma(T_O, dS + tc::koff(128, kk), (s ? dQK1 : dQK0) + tc::koff(128, kk), ID_N64, kk > 0);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        tc::mma(T_O, dVN + tc::koff(128, kk), (s ? dA1 : dA0) + tc::koff(64, kk), ID_N64, 1);
                }
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    tc::mma(T_DS, dVNd + tc::koff(128, kk), (s ? dKmn1 : dKmn0) + tc::mnoff(kk), ID_N128_BMN, kk > 0);
                tc::commit(&sm.mbar_s);
            }
            if (!(ok = wait_mma())) break;
            const float eglast = sm.slot[s].eglast;
            o_tb = sm.slot[s].tb;
            o_valid = sm.slot[s].valid;
            o_pending = job.write_o;
            tc::fence_before();
            tc::bar_sync(BAR_S, GS);
            if (gt == 0) tc::mbar_arrive(&sm.empty[s]);
            {  // S <- e^{G_last} S + dS
                float ds[32];
#pragma unroll
                for (int q2 = 0; q2 < 2; ++q2) {
                    tc::ld32(T_DS + lb + 64 * half + 32 * q2, ds);
#pragma unroll
                    for (int c2 = 0; c2 < 32; ++c2) Sr[32 * q2 + c2] = fmaf(eglast, Sr[32 * q2 + c2], ds[c2]);
                }
#pragma unroll
                for (int c8 = 0; c8 < 8; ++c8)
                    *reinterpret_cast<uint4*>(&sm.S[tc::sw128_chunk(128, row, 8 * half + c8)]) = pack8(&Sr[8 * c8]);
            }
            tc::fence_async_smem();
            tc::fence_before();
            tc::bar_sync(BAR_S, GS);
        }
        if (ok && o_pending) store_o(o_tb, o_valid);
        if (ok && job.fin) {
#pragma unroll
            for (int c2 = 0; c2 < 64; ++c2) job.fin[(int64_t)(64 * half + c2) * job.fin_ld + row] = Sr[c2];
        }
    }
    if (!ok && gt == 0) atomicAdd(&g_gdn_timeouts, 1);
    tc::fence_before();
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc(tmem, 512);
}

}  // namespace

gdn_status set_smem_attr(const void* func, size_t bytes);

bool chunk_tc_eligible(gdn_dtype dt, int dk, int dv) { return dt == GDN_BF16 && dk == 128 && dv == 128; }

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_tiled() {
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    }
    return fn;
}

// [rows x cols] bf16 view with row stride ld (elements), 64x64 boxes, 128B swizzle;
// rows past the end read as zero.
static gdn_status make_map(CUtensorMap* m, const void* base, int64_t ld, int64_t cols, int64_t rows) {
    EncodeTiledFn fn = encode_tiled();
    if (!fn) return fail(GDN_ERR_CUDA, "cuTensorMapEncodeTiled unavailable");
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)(rows > 0 ? rows : 1)};
    const cuuint64_t strides[1] = {(cuuint64_t)ld * 2};
    const cuuint32_t box[2] = {64, 64}, es[2] = {1, 1};
    const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(GDN_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
    return GDN_OK;
}

gdn_status launch_chunk_tc(const ChunkParams& p, int src, dim3 grid, cudaStream_t s) {
    const size_t smem = sizeof(SmemWS) + 1024;
    gdn_status st = set_smem_attr((const void*)chunk_tc_kernel, smem);
    if (st != GDN_OK) return st;
    TmaMaps maps;
    memset(&maps, 0, sizeof(maps));
    if (p.T > 0) {
        if ((st = make_map(&maps.q, p.q, p.ldq, (int64_t)p.Hk * 128, p.T)) != GDN_OK) return st;
        if ((st = make_map(&maps.k, p.k, p.ldk, (int64_t)p.Hk * 128, p.T)) != GDN_OK) return st;
        if ((st = make_map(&maps.v, p.v, p.ldv, (int64_t)p.Hv * 128, p.T)) != GDN_OK) return st;
    }
    chunk_tc_kernel<<<grid, NT, smem, s>>>(p, src, maps);
    return check_launch("chunk_tc_kernel");
}

}  // namespace gdn
