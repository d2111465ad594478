// bf16 chunk kernel (tensor cores via mma.sync m16n8k16, fp32 accumulate).
//
// One CTA (4 warps) runs one job: a token range of one value head and a tile
// of DVT state columns, chunk after chunk (C = 64).  Per chunk, warp w owns
// rows 16w..16w+15 of every [64 x *] product (Gram, W, U, v_new, o); the
// fp32 state S [DK x DVT] stays in registers as mma accumulators, split over
// the warps, with a bf16 copy in shared memory as the B operand of W S and
// Q S.  The 64x64 UT inverse runs in fp32 on the FFMA pipe.
#include "chunk_common.cuh"

namespace gdn {
namespace {

constexpr int NT = 128;
constexpr int LDF = 68;  // row stride (floats) of the 64x64 fp32 tiles
typedef __nv_bfloat16 bf16;

// XOR-swizzled bf16 tile with ROW elements per row: 16-byte chunk `ch` of row
// `r` is stored at chunk position ch ^ f(r), so that ldmatrix reads of 8 rows
// at one logical chunk hit 8 different bank groups.
template <int ROW>
__device__ __forceinline__ int swz(int r, int ch) {
    constexpr int CH = ROW / 8;
    const int x = (CH >= 8) ? (ch ^ (r & 7)) : (ch ^ ((r >> 1) & (CH - 1)));
    return r * ROW + x * 8;
}
template <int ROW>
__device__ __forceinline__ int swz_el(int r, int c) {
    return swz<ROW>(r, c >> 3) + (c & 7);
}

__device__ __forceinline__ void mma16816(float* c, const uint32_t* a, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void ldsm4(uint32_t* r, const void* p) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(smem_u32(p)));
}
__device__ __forceinline__ void ldsm4t(uint32_t* r, const void* p) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(smem_u32(p)));
}
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}

// A fragment (16x16) of a row-major [m][k] tile.
template <int ROW>
__device__ __forceinline__ void frag_a(uint32_t* a, const bf16* t, int m0, int k0) {
    const int l = threadIdx.x & 31;
    ldsm4(a, t + swz<ROW>(m0 + (l & 15), (k0 >> 3) + (l >> 4)));
}
// A fragment (16x16) of A = X^T where X is a row-major [k][m] tile.
template <int ROW>
__device__ __forceinline__ void frag_a_t(uint32_t* a, const bf16* t, int m0, int k0) {
    const int l = threadIdx.x & 31;
    ldsm4t(a, t + swz<ROW>(k0 + ((l >> 4) << 3) + (l & 7), (m0 >> 3) + ((l >> 3) & 1)));
}
// B fragments for two n8 tiles (k16 x n16) of B = X^T, X row-major [n][k].
template <int ROW>
__device__ __forceinline__ void frag_b_nk(uint32_t* b, const bf16* t, int n0, int k0) {
    const int l = threadIdx.x & 31;
    ldsm4(b, t + swz<ROW>(n0 + (l & 7) + ((l >> 4) << 3), (k0 >> 3) + ((l >> 3) & 1)));
}
// B fragments for two n8 tiles (k16 x n16) of a row-major [k][n] tile.
template <int ROW>
__device__ __forceinline__ void frag_b_kn(uint32_t* b, const bf16* t, int k0, int n0) {
    const int l = threadIdx.x & 31;
    ldsm4t(b, t + swz<ROW>(k0 + (l & 7) + (((l >> 3) & 1) << 3), (n0 >> 3) + (l >> 4)));
}

template <int DK, int DVT>
struct SmemB {
    bf16 Q[64 * DK];
    bf16 K[64 * DK];
    bf16 S[DK * DVT];      // bf16 copy of the state (B operand)
    bf16 VO[64 * DVT];     // value tile; later the output staging tile
    union {
        float L[64 * LDF]; // strictly lower L (dead after the inverse)
        struct {
            bf16 VN[64 * DVT];   // v_new
            bf16 VNd[64 * DVT];  // v_new scaled by exp(G_last - G_i)
        } vn;
    } u;
    float Tm[64 * LDF];
    float X[3 * 16 * 17];
    float g[64], beta[64], G[64], eG[64], eGl[64];
};

template <int DK, int DVT>
__global__ void __launch_bounds__(NT, 2) chunk_bf16_kernel(const ChunkParams p, const int src) {
    extern __shared__ __align__(128) unsigned char smem_raw[];
    SmemB<DK, DVT>& sm = *reinterpret_cast<SmemB<DK, DVT>*>(smem_raw);
    ChunkJob job;
    if (!make_job(p, src, job)) return;

    const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
    const int g8 = lane >> 2, tq = lane & 3;
    const int hv = job.hv, hk = hv / (p.Hv / p.Hk);
    const bf16* __restrict__ q = static_cast<const bf16*>(p.q);
    const bf16* __restrict__ k = static_cast<const bf16*>(p.k);
    const bf16* __restrict__ v = static_cast<const bf16*>(p.v);
    bf16* __restrict__ o = static_cast<bf16*>(p.o);
    const bool l2 = (p.flags & GDN_QK_L2NORM) != 0;

    // state ownership: SWR x SWC warps over [DK x DVT]
    constexpr int SWR = (DK / 16 < 4) ? DK / 16 : 4;
    constexpr int SWC = 4 / SWR;
    constexpr int RS = DK / SWR, CS = DVT / SWC;
    constexpr int SMT = RS / 16, SNT = CS / 8;
    static_assert(SNT % 2 == 0, "state column tile");
    const int srow0 = (w / SWC) * RS, scol0 = (w % SWC) * CS;

    float accS[SMT][SNT][4];
#pragma unroll
    for (int mt = 0; mt < SMT; ++mt)
#pragma unroll
        for (int nt = 0; nt < SNT; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int r = srow0 + mt * 16 + g8 + ((e >> 1) << 3);
                const int c = scol0 + nt * 8 + 2 * tq + (e & 1);
                float s0 = 0.f;
                if (job.identity_init) s0 = (r == job.col0 + c) ? 1.f : 0.f;
                else if (job.init) s0 = job.init[(int64_t)r * job.init_ld + c];
                accS[mt][nt][e] = s0;
            }
#pragma unroll
    for (int mt = 0; mt < SMT; ++mt)
#pragma unroll
        for (int nt = 0; nt < SNT; ++nt) {
            const int r = srow0 + mt * 16 + g8;
            const int c = scol0 + nt * 8 + 2 * tq;
            *reinterpret_cast<uint32_t*>(&sm.S[swz_el<DVT>(r, c)]) = pack2(accS[mt][nt][0], accS[mt][nt][1]);
            *reinterpret_cast<uint32_t*>(&sm.S[swz_el<DVT>(r + 8, c)]) = pack2(accS[mt][nt][2], accS[mt][nt][3]);
        }

    const int nch = (job.t1 - job.t0 + 63) / 64;
    for (int ch = 0; ch < nch; ++ch) {
        const int tb = job.t0 + ch * 64;
        const int valid = min(64, job.t1 - tb);
        __syncthreads();
        // ---- load the chunk (rows past the end read as zero) ----
        constexpr int QCH = DK / 8;
        for (int e = tid; e < 64 * QCH; e += NT) {
            const int r = e / QCH, c8 = e % QCH;
            const int64_t t = tb + (r < valid ? r : 0);
            const int nb = r < valid ? 16 : 0;
            cp_async16(&sm.Q[swz<DK>(r, c8)], q + t * p.ldq + (int64_t)hk * p.hsq + c8 * 8, nb);
            cp_async16(&sm.K[swz<DK>(r, c8)], k + t * p.ldk + (int64_t)hk * p.hsk + c8 * 8, nb);
        }
        if (!job.value_zero) {
            constexpr int VCH = DVT / 8;
            for (int e = tid; e < 64 * VCH; e += NT) {
                const int r = e / VCH, c8 = e % VCH;
                const int64_t t = tb + (r < valid ? r : 0);
                cp_async16(&sm.VO[swz<DVT>(r, c8)],
                           v + t * p.ldv + (int64_t)hv * p.hsv + job.col0 + c8 * 8, r < valid ? 16 : 0);
            }
        }
        cp_async_commit();
        if (tid < 64) {
            const int64_t t = tb + tid;
            float gv = 0.f, bv = 0.f;
            if (tid < valid) gate_beta<bf16>(p, t, hv, gv, bv);
            sm.g[tid] = gv;
            sm.beta[tid] = bv;
        }
        cp_async_wait_all();
        __syncthreads();
        if (l2) {
            // q, k <- x * rsqrt(|x|^2 + 1e-6): QCH lanes per row, one 16-byte chunk each
            constexpr int RPI = 32 / QCH;  // rows per warp iteration
            const int sub = lane / QCH, c8 = lane % QCH;
            for (int r0 = w * RPI; r0 < 128; r0 += 4 * RPI) {
                const int r = r0 + sub;
                bf16* tile = r < 64 ? sm.Q : sm.K;
                const int rr = r & 63;
                uint4* ptr = reinterpret_cast<uint4*>(&tile[swz<DK>(rr, c8)]);
                uint4 raw = *ptr;
                __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&raw);
                float f[8];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    float2 t2 = __bfloat1622float2(h[i]);
                    f[2 * i] = t2.x;
                    f[2 * i + 1] = t2.y;
                }
                float ss = 0.f;
#pragma unroll
                for (int i = 0; i < 8; ++i) ss = fmaf(f[i], f[i], ss);
#pragma unroll
                for (int off = QCH / 2; off; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
                const float rn = rsqrtf(ss + 1e-6f);
#pragma unroll
                for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(f[2 * i] * rn, f[2 * i + 1] * rn);
                *ptr = raw;
            }
        }
        if (w == 0) gate_prefix_warp0(sm.g, sm.G, sm.eG, sm.eGl);
        __syncthreads();

        // ---- Gram products for rows 16w..16w+15: K K^T and Q K^T (causal half) ----
        float kk[8][4], qk[8][4];
#pragma unroll
        for (int nt = 0; nt < 8; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) kk[nt][e] = qk[nt][e] = 0.f;
#pragma unroll
        for (int kt = 0; kt < DK / 16; ++kt) {
            uint32_t ak[4], aq[4];
            frag_a<DK>(ak, sm.K, 16 * w, 16 * kt);
            frag_a<DK>(aq, sm.Q, 16 * w, 16 * kt);
#pragma unroll
            for (int np = 0; np < 4; ++np) {
                if (np <= w) {
                    uint32_t b[4];
                    frag_b_nk<DK>(b, sm.K, 16 * np, 16 * kt);
                    mma16816(kk[2 * np], ak, b[0], b[1]);
                    mma16816(kk[2 * np + 1], ak, b[2], b[3]);
                    mma16816(qk[2 * np], aq, b[0], b[1]);
                    mma16816(qk[2 * np + 1], aq, b[2], b[3]);
                }
            }
        }
        // L -> shared (fp32); A = scale Q K^T o Gamma -> bf16 A fragments
        uint32_t aqf[4][4];
        {
            const int i0 = 16 * w + g8, i1 = i0 + 8;
            const float G0 = sm.G[i0], G1 = sm.G[i1], b0 = sm.beta[i0], b1 = sm.beta[i1];
            float av[8][4];
#pragma unroll
            for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int i = (e >> 1) ? i1 : i0;
                    const int j = nt * 8 + 2 * tq + (e & 1);
                    const float Gi = (e >> 1) ? G1 : G0;
                    const float gam = (i >= j) ? __expf(Gi - sm.G[j]) : 0.f;
                    sm.u.L[i * LDF + j] = (i > j) ? ((e >> 1) ? b1 : b0) * kk[nt][e] * gam : 0.f;
                    av[nt][e] = p.scale * qk[nt][e] * gam;
                }
            }
#pragma unroll
            for (int kt = 0; kt < 4; ++kt) {
                aqf[kt][0] = pack2(av[2 * kt][0], av[2 * kt][1]);
                aqf[kt][1] = pack2(av[2 * kt][2], av[2 * kt][3]);
                aqf[kt][2] = pack2(av[2 * kt + 1][0], av[2 * kt + 1][1]);
                aqf[kt][3] = pack2(av[2 * kt + 1][2], av[2 * kt + 1][3]);
            }
        }
        __syncthreads();
        unit_lower_inverse64<NT, LDF>(sm.u.L, sm.Tm, sm.X);

        // ---- W = T diag(beta e^G) K, U = T diag(beta) V  (rows 16w..) ----
        float wacc[DK / 8][4];
        float uacc[DVT / 8][4];
#pragma unroll
        for (int nt = 0; nt < DK / 8; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) wacc[nt][e] = 0.f;
#pragma unroll
        for (int nt = 0; nt < DVT / 8; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) uacc[nt][e] = 0.f;
        {
            const int i0 = 16 * w + g8, i1 = i0 + 8;
#pragma unroll
            for (int kt = 0; kt < 4; ++kt) {
                if (kt <= w) {
                    const int j0 = 16 * kt + 2 * tq;
                    const float2 t00 = *reinterpret_cast<const float2*>(&sm.Tm[i0 * LDF + j0]);
                    const float2 t10 = *reinterpret_cast<const float2*>(&sm.Tm[i1 * LDF + j0]);
                    const float2 t01 = *reinterpret_cast<const float2*>(&sm.Tm[i0 * LDF + j0 + 8]);
                    const float2 t11 = *reinterpret_cast<const float2*>(&sm.Tm[i1 * LDF + j0 + 8]);
                    const float bv0 = sm.beta[j0], bv1 = sm.beta[j0 + 1];
                    const float bv8 = sm.beta[j0 + 8], bv9 = sm.beta[j0 + 9];
                    const float bw0 = bv0 * sm.eG[j0], bw1 = bv1 * sm.eG[j0 + 1];
                    const float bw8 = bv8 * sm.eG[j0 + 8], bw9 = bv9 * sm.eG[j0 + 9];
                    uint32_t aw[4] = {pack2(t00.x * bw0, t00.y * bw1), pack2(t10.x * bw0, t10.y * bw1),
                                      pack2(t01.x * bw8, t01.y * bw9), pack2(t11.x * bw8, t11.y * bw9)};
#pragma unroll
                    for (int dn = 0; dn < DK / 16; ++dn) {
                        uint32_t b[4];
                        frag_b_kn<DK>(b, sm.K, 16 * kt, 16 * dn);
                        mma16816(wacc[2 * dn], aw, b[0], b[1]);
                        mma16816(wacc[2 * dn + 1], aw, b[2], b[3]);
                    }
                    if (!job.value_zero) {
                        uint32_t au[4] = {pack2(t00.x * bv0, t00.y * bv1), pack2(t10.x * bv0, t10.y * bv1),
                                          pack2(t01.x * bv8, t01.y * bv9), pack2(t11.x * bv8, t11.y * bv9)};
#pragma unroll
                        for (int vn = 0; vn < DVT / 16; ++vn) {
                            uint32_t b[4];
                            frag_b_kn<DVT>(b, sm.VO, 16 * kt, 16 * vn);
                            mma16816(uacc[2 * vn], au, b[0], b[1]);
                            mma16816(uacc[2 * vn + 1], au, b[2], b[3]);
                        }
                    }
                }
            }
        }
        // ---- v_new = U - W S ----
#pragma unroll
        for (int kt = 0; kt < DK / 16; ++kt) {
            uint32_t a[4] = {pack2(-wacc[2 * kt][0], -wacc[2 * kt][1]),
                             pack2(-wacc[2 * kt][2], -wacc[2 * kt][3]),
                             pack2(-wacc[2 * kt + 1][0], -wacc[2 * kt + 1][1]),
                             pack2(-wacc[2 * kt + 1][2], -wacc[2 * kt + 1][3])};
#pragma unroll
            for (int vn = 0; vn < DVT / 16; ++vn) {
                uint32_t b[4];
                frag_b_kn<DVT>(b, sm.S, 16 * kt, 16 * vn);
                mma16816(uacc[2 * vn], a, b[0], b[1]);
                mma16816(uacc[2 * vn + 1], a, b[2], b[3]);
            }
        }
        {
            const int i0 = 16 * w + g8, i1 = i0 + 8;
            const float d0 = sm.eGl[i0], d1 = sm.eGl[i1];
#pragma unroll
            for (int nt = 0; nt < DVT / 8; ++nt) {
                const int c = nt * 8 + 2 * tq;
                *reinterpret_cast<uint32_t*>(&sm.u.vn.VN[swz_el<DVT>(i0, c)]) = pack2(uacc[nt][0], uacc[nt][1]);
                *reinterpret_cast<uint32_t*>(&sm.u.vn.VN[swz_el<DVT>(i1, c)]) = pack2(uacc[nt][2], uacc[nt][3]);
                *reinterpret_cast<uint32_t*>(&sm.u.vn.VNd[swz_el<DVT>(i0, c)]) =
                    pack2(uacc[nt][0] * d0, uacc[nt][1] * d0);
                *reinterpret_cast<uint32_t*>(&sm.u.vn.VNd[swz_el<DVT>(i1, c)]) =
                    pack2(uacc[nt][2] * d1, uacc[nt][3] * d1);
            }
        }
        __syncthreads();

        // ---- o = scale e^G (Q S) + A v_new ----
        if (job.write_o) {
            float oacc[DVT / 8][4];
#pragma unroll
            for (int nt = 0; nt < DVT / 8; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) oacc[nt][e] = 0.f;
#pragma unroll
            for (int kt = 0; kt < DK / 16; ++kt) {
                uint32_t a[4];
                frag_a<DK>(a, sm.Q, 16 * w, 16 * kt);
#pragma unroll
                for (int vn = 0; vn < DVT / 16; ++vn) {
                    uint32_t b[4];
                    frag_b_kn<DVT>(b, sm.S, 16 * kt, 16 * vn);
                    mma16816(oacc[2 * vn], a, b[0], b[1]);
                    mma16816(oacc[2 * vn + 1], a, b[2], b[3]);
                }
            }
            const int i0 = 16 * w + g8, i1 = i0 + 8;
            const float f0 = p.scale * sm.eG[i0], f1 = p.scale * sm.eG[i1];
#pragma unroll
            for (int nt = 0; nt < DVT / 8; ++nt) {
                oacc[nt][0] *= f0; oacc[nt][1] *= f0;
                oacc[nt][2] *= f1; oacc[nt][3] *= f1;
            }
#pragma unroll
            for (int kt = 0; kt < 4; ++kt) {
                if (kt <= w) {
#pragma unroll
                    for (int vn = 0; vn < DVT / 16; ++vn) {
                        uint32_t b[4];
                        frag_b_kn<DVT>(b, sm.u.vn.VN, 16 * kt, 16 * vn);
                        mma16816(oacc[2 * vn], aqf[kt], b[0], b[1]);
                        mma16816(oacc[2 * vn + 1], aqf[kt], b[2], b[3]);
                    }
                }
            }
#pragma unroll
            for (int nt = 0; nt < DVT / 8; ++nt) {
                const int c = nt * 8 + 2 * tq;
                *reinterpret_cast<uint32_t*>(&sm.VO[swz_el<DVT>(i0, c)]) = pack2(oacc[nt][0], oacc[nt][1]);
                *reinterpret_cast<uint32_t*>(&sm.VO[swz_el<DVT>(i1, c)]) = pack2(oacc[nt][2], oacc[nt][3]);
            }
        }
        __syncthreads();
        if (job.write_o) {
            constexpr int VCH = DVT / 8;
            for (int e = tid; e < 64 * VCH; e += NT) {
                const int r = e / VCH, c8 = e % VCH;
                if (r < valid) {
                    *reinterpret_cast<uint4*>(o + (int64_t)(tb + r) * p.ldo + (int64_t)hv * p.hso + job.col0 + c8 * 8) =
                        *reinterpret_cast<const uint4*>(&sm.VO[swz<DVT>(r, c8)]);
                }
            }
        }

        // ---- S <- e^{G_last} S + K^T (v_new o e^{G_last - G}) ----
        const float eGlast = sm.eG[63];
#pragma unroll
        for (int mt = 0; mt < SMT; ++mt)
#pragma unroll
            for (int nt = 0; nt < SNT; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) accS[mt][nt][e] *= eGlast;
#pragma unroll
        for (int kt = 0; kt < 4; ++kt) {
#pragma unroll
            for (int mt = 0; mt < SMT; ++mt) {
                uint32_t a[4];
                frag_a_t<DK>(a, sm.K, srow0 + 16 * mt, 16 * kt);
#pragma unroll
                for (int n2 = 0; n2 < SNT / 2; ++n2) {
                    uint32_t b[4];
                    frag_b_kn<DVT>(b, sm.u.vn.VNd, 16 * kt, scol0 + 16 * n2);
                    mma16816(accS[mt][2 * n2], a, b[0], b[1]);
                    mma16816(accS[mt][2 * n2 + 1], a, b[2], b[3]);
                }
            }
        }
#pragma unroll
        for (int mt = 0; mt < SMT; ++mt)
#pragma unroll
            for (int nt = 0; nt < SNT; ++nt) {
                const int r = srow0 + mt * 16 + g8;
                const int c = scol0 + nt * 8 + 2 * tq;
                *reinterpret_cast<uint32_t*>(&sm.S[swz_el<DVT>(r, c)]) = pack2(accS[mt][nt][0], accS[mt][nt][1]);
                *reinterpret_cast<uint32_t*>(&sm.S[swz_el<DVT>(r + 8, c)]) = pack2(accS[mt][nt][2], accS[mt][nt][3]);
            }
    }
    if (job.fin) {
#pragma unroll
        for (int mt = 0; mt < SMT; ++mt)
#pragma unroll
            for (int nt = 0; nt < SNT; ++nt) {
                const int r = srow0 + mt * 16 + g8;
                const int c = scol0 + nt * 8 + 2 * tq;
                *reinterpret_cast<float2*>(job.fin + (int64_t)r * job.fin_ld + c) =
                    make_float2(accS[mt][nt][0], accS[mt][nt][1]);
                *reinterpret_cast<float2*>(job.fin + (int64_t)(r + 8) * job.fin_ld + c) =
                    make_float2(accS[mt][nt][2], accS[mt][nt][3]);
            }
    }
}

}  // namespace

gdn_status set_smem_attr(const void* func, size_t bytes);

template <int DK, int DVT>
static gdn_status launch_t(const ChunkParams& p, int src, dim3 grid, cudaStream_t s) {
    const size_t smem = sizeof(SmemB<DK, DVT>);
    gdn_status st = set_smem_attr((const void*)chunk_bf16_kernel<DK, DVT>, smem);
    if (st != GDN_OK) return st;
    chunk_bf16_kernel<DK, DVT><<<grid, NT, smem, s>>>(p, src);
    return check_launch("chunk_bf16_kernel");
}

gdn_status launch_chunk_bf16(const ChunkParams& p, int src, dim3 grid, cudaStream_t s) {
    if (p.col_tile == 64) {
        switch (p.dk) {
            case 32: return launch_t<32, 64>(p, src, grid, s);
            case 64: return launch_t<64, 64>(p, src, grid, s);
            case 128: return launch_t<128, 64>(p, src, grid, s);
        }
    } else if (p.col_tile == 32) {
        switch (p.dk) {
            case 32: return launch_t<32, 32>(p, src, grid, s);
            case 64: return launch_t<64, 32>(p, src, grid, s);
            case 128: return launch_t<128, 32>(p, src, grid, s);
        }
    }
    return fail(GDN_ERR_UNSUPPORTED_SHAPE, "bf16 chunk: dk=%d col_tile=%d", p.dk, p.col_tile);
}

}  // namespace gdn
