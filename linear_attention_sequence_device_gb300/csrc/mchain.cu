// The M chain of the shard summaries on the tensor cores (hyper-parallel page
// linear_attention_context_parallel.py: _compute_gdn_state_summary_from_prepared,
// the transition product M <- M_i M with M_i = e^{G_C} I - Kd^T W).
//
// In shard pass 1 the N job of every spanning shard stores, per chunk, the
// bf16 W rows and K~ tile it built for its own chain, and e^{G_last}.  The M
// chain of the same shard needs exactly those operands and no value input, so
// this kernel runs it on its own, from the identity, with the chunk kernel's
// products and state handling (M comes out as the chunk kernel's M job would
// give it):
//   v_new^T = -S^T W^T,   S^T <- e^{G_last} S^T + v_new^T K~.
// One CTA of 128 threads per (shard, value head, segment); thread =
// tensor-memory lane = row of S^T.  It holds 256 tensor-memory columns, so two
// CTAs share an SM and their chains interleave.  The next chunk's W / K~ load
// (TMA) while the current one runs.  Every wait is bounded: on expiry the
// kernel counts a timeout, writes GDN_ERR_TIMEOUT to the plan's status word
// and leaves.
//
// When there are fewer chains than resident CTAs (few long shards), each chain
// is cut into G segments run side by side, each from the identity; M is the
// ordered product of the segments' transitions (the product is associative),
// formed in fp32 by mchain_merge_kernel.
#include <cuda.h>
#include <string.h>

#include "gdn_internal.cuh"
#include "tc_util.cuh"

namespace gdn {

extern __device__ int g_gdn_timeouts;
gdn_status make_map_bf16(CUtensorMap* m, const void* base, int64_t ld, int64_t cols, int64_t rows);
gdn_status set_smem_attr(const void* func, size_t bytes);

namespace {

constexpr int MT = 128;
inline size_t al256(size_t x) { return (x + 255) & ~(size_t)255; }
constexpr uint32_t kMSpin = 1u << 20;
constexpr size_t kMSmemFloor = 96 * 1024;  // shared memory that leaves room for two CTAs an SM, not three
constexpr int BAR_M = 1;
typedef __nv_bfloat16 bf16;

struct MMaps {
    CUtensorMap w, kt;  // [chunks * 64 rows x 128 columns] bf16, 64x64 boxes, 128-byte swizzle
};

struct MParams {
    const int32_t* plan;
    int num_seqs, P, Hv, nch;  // nch: chunks of a shard
    const float* eg;            // e^{G_last} of every stored chunk
    float* M;                   // [P, Hv, 128, 128]: M of shard r at r
    float* Mseg;                // [P, Hv, G, 128, 128]: the segments' products (G > 1)
};

struct MSmem {
    bf16 W[2][64 * 128];   // per stage: W rows [token][key], K-major (two 64-key atoms)
    bf16 KT[2][64 * 128];  // per stage: K~ [token][key], MN-major (two 64-key atoms)
    uint64_t ld[2];        // TMA arrivals
    uint64_t mma;          // product completions
    uint64_t fin;
    int issued[2], waited[2];
    uint32_t tmem_slot;
};

// 32 lanes x 64 consecutive 32-bit columns in one tensor-memory access (one
// wait for all 64 loads): the state read-back takes two of these per thread.
__device__ __forceinline__ void ld64(uint32_t taddr, float* v) {
    uint32_t r[64];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x64.b32 {"
        "%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,"
        "%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,"
        "%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63"
        "}, [%64];\n"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]),
          "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]),
          "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]),
          "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]),
          "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int i = 0; i < 64; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void st64(uint32_t taddr, const float* v) {
    uint32_t u[64];
#pragma unroll
    for (int i = 0; i < 64; ++i) u[i] = __float_as_uint(v[i]);
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x64.b32 [%0], {"
        "%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,"
        "%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,"
        "%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63,%64"
        "};"
        :
        : "r"(taddr),
          "r"(u[0]), "r"(u[1]), "r"(u[2]), "r"(u[3]), "r"(u[4]), "r"(u[5]), "r"(u[6]), "r"(u[7]),
          "r"(u[8]), "r"(u[9]), "r"(u[10]), "r"(u[11]), "r"(u[12]), "r"(u[13]), "r"(u[14]), "r"(u[15]),
          "r"(u[16]), "r"(u[17]), "r"(u[18]), "r"(u[19]), "r"(u[20]), "r"(u[21]), "r"(u[22]), "r"(u[23]),
          "r"(u[24]), "r"(u[25]), "r"(u[26]), "r"(u[27]), "r"(u[28]), "r"(u[29]), "r"(u[30]), "r"(u[31]),
          "r"(u[32]), "r"(u[33]), "r"(u[34]), "r"(u[35]), "r"(u[36]), "r"(u[37]), "r"(u[38]), "r"(u[39]),
          "r"(u[40]), "r"(u[41]), "r"(u[42]), "r"(u[43]), "r"(u[44]), "r"(u[45]), "r"(u[46]), "r"(u[47]),
          "r"(u[48]), "r"(u[49]), "r"(u[50]), "r"(u[51]), "r"(u[52]), "r"(u[53]), "r"(u[54]), "r"(u[55]),
          "r"(u[56]), "r"(u[57]), "r"(u[58]), "r"(u[59]), "r"(u[60]), "r"(u[61]), "r"(u[62]), "r"(u[63])
        : "memory");
}
__device__ __forceinline__ void stw32(uint32_t taddr, const uint32_t* w) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {"
        "%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32"
        "};"
        :
        : "r"(taddr),
          "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7]),
          "r"(w[8]), "r"(w[9]), "r"(w[10]), "r"(w[11]), "r"(w[12]), "r"(w[13]), "r"(w[14]), "r"(w[15]),
          "r"(w[16]), "r"(w[17]), "r"(w[18]), "r"(w[19]), "r"(w[20]), "r"(w[21]), "r"(w[22]), "r"(w[23]),
          "r"(w[24]), "r"(w[25]), "r"(w[26]), "r"(w[27]), "r"(w[28]), "r"(w[29]), "r"(w[30]), "r"(w[31])
        : "memory");
}

constexpr uint32_t ID_N64_NEG = tc::idesc_bf16(128, 64, false, false, false) | (1u << 14);
constexpr uint32_t ID_N128_BMN = tc::idesc_bf16(128, 128, false, true, false);

__global__ void __launch_bounds__(MT) mchain_kernel(const MParams p, const __grid_constant__ MMaps maps) {
    extern __shared__ unsigned char smem_raw[];
    MSmem& sm = *reinterpret_cast<MSmem*>(smem_raw + ((1024 - (tc::smem_addr(smem_raw) & 1023)) & 1023));
    const int r = blockIdx.x, hv = blockIdx.y, z = blockIdx.z, G = gridDim.z, tid = threadIdx.x, warp = tid >> 5;
    if (__ldg(p.plan) != 0) return;  // malformed cu_seqlens: nothing to do
    // a spanning shard: one local segment, continued from and into its neighbours
    const int32_t* rec = p.plan + 1 + (int64_t)r * GDN_PLAN_NFIELDS;
    if (!(__ldg(rec + GDN_PLAN_LOCAL_NUM_SEQS) == 1 && !__ldg(rec + GDN_PLAN_IS_FIRST_RANK) &&
          __ldg(rec + GDN_PLAN_POST_NUM_RANKS) > 0))
        return;
    const int nch = p.nch;
    const int c0 = (int)((int64_t)z * nch / G), c1 = (int)((int64_t)(z + 1) * nch / G);  // this segment's chunks
    if (c1 <= c0) return;
    const int64_t item = (int64_t)r * p.Hv + hv;
    const int y0 = (int)(item * nch * 64);  // first stored row of this shard's chunks
    const float* eg = p.eg + item * nch;

    if (tid == 0) {
        tc::mbar_init(&sm.ld[0], 1);
        tc::mbar_init(&sm.ld[1], 1);
        tc::mbar_init(&sm.mma, 1);
        tc::mbar_init(&sm.fin, 1);
        sm.issued[0] = sm.issued[1] = sm.waited[0] = sm.waited[1] = 0;
    }
    tc::fence_async_smem();
    if (warp == 0) tc::tmem_alloc(&sm.tmem_slot, 256);
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tmem = sm.tmem_slot;
    // columns: fp32 S^T | bf16 S^T (two keys per column) | v_new (fp32, then bf16 pairs in place)
    const uint32_t lb = (uint32_t)(warp * 32) << 16;
    const uint32_t T_S = tmem + lb, T_SB = tmem + 128 + lb, T_VN = tmem + 192 + lb;
    const int row = tid;  // tensor-memory lane = row of S^T

    auto issue_load = [&](int c) {  // W rows and K~ of chunk c into stage (c - c0) & 1 (thread 0)
        const int st = (c - c0) & 1, y = y0 + 64 * c;
        tc::mbar_expect_tx(&sm.ld[st], 4 * 64 * 64 * 2);
        tc::tma_load_2d(sm.W[st], &maps.w, 0, y, &sm.ld[st]);
        tc::tma_load_2d(sm.W[st] + 64 * 64, &maps.w, 64, y, &sm.ld[st]);
        tc::tma_load_2d(sm.KT[st], &maps.kt, 0, y, &sm.ld[st]);
        tc::tma_load_2d(sm.KT[st] + 64 * 64, &maps.kt, 64, y, &sm.ld[st]);
        sm.issued[st] += 1;
    };
    if (tid == 0) {
        issue_load(c0);
        if (c0 + 1 < c1) issue_load(c0 + 1);
    }
    // the identity, as bf16 (the first product's A operand) and scaled by the
    // first chunk's e^{G_last} (the first update accumulates onto it)
    {
        const float e0 = __ldg(eg + c0);
#pragma unroll 1
        for (int h = 0; h < 2; ++h)
#pragma unroll 1
            for (int q4 = 0; q4 < 4; ++q4) {
                float v[16];
                uint32_t w[8];
#pragma unroll
                for (int c2 = 0; c2 < 16; ++c2) v[c2] = (64 * h + 16 * q4 + c2 == row) ? 1.f : 0.f;
#pragma unroll
                for (int j = 0; j < 8; ++j) w[j] = tc::pack_bf16x2(v[2 * j], v[2 * j + 1]);
                tc::stw8(T_SB + 32 * h + 8 * q4, w);
#pragma unroll
                for (int c2 = 0; c2 < 16; ++c2) v[c2] *= e0;
                tc::st16(T_S + 64 * h + 16 * q4, v);
            }
    }
    const uint64_t dW0 = tc::desc(tc::smem_addr(sm.W[0]), 16, 1024);
    const uint64_t dKT0 = tc::desc(tc::smem_addr(sm.KT[0]), 64 * 128, 1024);
    constexpr uint64_t kStage = sizeof(bf16) * 64 * 128 / 16;  // descriptor start-address step of a stage
    uint32_t ph = 0;
    bool ok = true;
    auto wait_mma = [&]() -> bool {
        bool d = true;
        if (tid == 0) d = tc::mbar_wait(&sm.mma, ph, kMSpin);
        ph ^= 1u;
        const bool all = tc::bar_and(BAR_M, MT, d);
        tc::fence_after();
        return all;
    };
    for (int c = c0; c < c1 && ok; ++c) {
        const int st = (c - c0) & 1;
        tc::st32_zero(T_VN);  // v_new = 0 - S^T W^T: the product accumulates onto zero
        tc::st32_zero(T_VN + 32);
        bool in = true;
        if (tid == 0) {
            in = tc::mbar_wait(&sm.ld[st], ((c - c0) >> 1) & 1, kMSpin);
            if (in) sm.waited[st] += 1;
        }
        tc::wait_st();
        tc::fence_before();
        if (!(ok = tc::bar_and(BAR_M, MT, in))) break;
        if (tid == 0) {
            tc::fence_after();
            const uint64_t dW = dW0 + (st ? kStage : 0);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) tc::mma_ta(T_VN - lb, T_SB - lb + 8 * kk, dW + tc::koff(64, kk), ID_N64_NEG, 1u);
            tc::commit(&sm.mma);
        }
        if (!(ok = wait_mma())) break;
        // v_new^T as bf16 pairs in place (the second product's A operand)
        {
            float vv[64];
            uint32_t w[32];
            ld64(T_VN, vv);
#pragma unroll
            for (int j = 0; j < 32; ++j) w[j] = tc::pack_bf16x2(vv[2 * j], vv[2 * j + 1]);
            tc::stw16(T_VN, w);
            tc::stw16(T_VN + 32, w + 16);
        }
        tc::wait_st();
        tc::fence_before();
        tc::bar_sync(BAR_M, MT);
        if (tid == 0) {
            tc::fence_after();
            const uint64_t dKT = dKT0 + (st ? kStage : 0);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                tc::mma_ta(T_S - lb, T_VN - lb + 32 * (kk >> 1) + 8 * (kk & 1), dKT + tc::mnoff(kk), ID_N128_BMN, 1u);
            tc::commit(&sm.mma);
        }
        if (!(ok = wait_mma())) break;
        if (tid == 0 && c + 2 < c1) issue_load(c + 2);  // both products of chunk c have read the stage
        if (c + 1 < c1) {
            // the new state: its bf16 copy, and the state scaled by the next
            // chunk's e^{G_last}, back into tensor memory
            const float egn = __ldg(eg + c + 1);
#pragma unroll 1
            for (int h = 0; h < 2; ++h) {  // 64 columns at a time: one load wait each
                float sv[64];
                uint32_t w[32];
                ld64(T_S + 64 * h, sv);
#pragma unroll
                for (int j = 0; j < 32; ++j) w[j] = tc::pack_bf16x2(sv[2 * j], sv[2 * j + 1]);
                stw32(T_SB + 32 * h, w);
#pragma unroll
                for (int c2 = 0; c2 < 64; ++c2) sv[c2] *= egn;
                st64(T_S + 64 * h, sv);
            }
        } else {
            float* fin = G > 1 ? p.Mseg + (item * G + z) * 128 * 128 : p.M + item * 128 * 128;
#pragma unroll 1
            for (int h = 0; h < 2; ++h)
#pragma unroll 1
                for (int q4 = 0; q4 < 4; ++q4) {
                    float v[16];
                    tc::ld16(T_S + 64 * h + 16 * q4, v);
#pragma unroll
                    for (int c2 = 0; c2 < 16; ++c2) fin[(int64_t)(64 * h + 16 * q4 + c2) * 128 + row] = v[c2];
                }
        }
    }
    if (!ok && tid == 0) {
        atomicAdd(&g_gdn_timeouts, 1);
        atomicCAS(const_cast<int32_t*>(p.plan), 0, (int)GDN_ERR_TIMEOUT);
    }
    if (tid == 0) {  // the products this thread issued and the loads still in flight are done
        tc::commit(&sm.fin);
        tc::mbar_wait(&sm.fin, 0, kMSpin);
        for (int st = 0; st < 2; ++st)
            if (sm.issued[st] > sm.waited[st]) tc::mbar_wait(&sm.ld[st], (sm.issued[st] - 1) & 1, kMSpin);
    }
    tc::fence_before();
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc(tmem, 256);
}

// M of every spanning shard from its G segments' products, each stored as
// the transpose of its S^T product: M = Mseg[G-1] ... Mseg[0], in fp32.  CTA
// (shard * Hv + head, block of 32 rows of M), 256 threads: warp w holds rows
// [4w, 4w + 4) of the block and lane l columns [4l, 4l + 4), a 4 x 4 tile of
// registers.  The running rows (transposed: a column of four rows is one
// 16-byte load) and each factor are staged in shared memory by coalesced
// loads, all in flight at once.
constexpr int kMergeRows = 32;
constexpr int kRt = 36;  // float stride of a transposed column (16-byte aligned, fewer bank conflicts)
constexpr size_t kMergeSmem = (size_t)(128 * kRt + 128 * 128) * sizeof(float);
__global__ void __launch_bounds__(256) mchain_merge_kernel(const int32_t* plan, int Hv, int G, const float* Mseg,
                                                           float* M) {
    extern __shared__ float4 merge_smem[];
    float* Rt = reinterpret_cast<float*>(merge_smem);  // [128 columns][kRt]: running rows, transposed
    float* F = Rt + 128 * kRt;                          // [128][128] factor
    const int64_t item = blockIdx.x;
    const int rb = blockIdx.y, tid = threadIdx.x;
    if (__ldg(plan) != 0) return;
    const int32_t* rec = plan + 1 + (item / Hv) * GDN_PLAN_NFIELDS;
    if (!(__ldg(rec + GDN_PLAN_LOCAL_NUM_SEQS) == 1 && !__ldg(rec + GDN_PLAN_IS_FIRST_RANK) &&
          __ldg(rec + GDN_PLAN_POST_NUM_RANKS) > 0))
        return;
    const float* seg = Mseg + item * G * 128 * 128;
    {
        const float4* src = reinterpret_cast<const float4*>(seg + (int64_t)(G - 1) * 128 * 128 + kMergeRows * rb * 128);
#pragma unroll
        for (int e0 = 0; e0 < kMergeRows * 32; e0 += 256) {
            const int e = e0 + tid, r = e >> 5, c = 4 * (e & 31);
            const float4 v = __ldg(src + e);
            Rt[(c + 0) * kRt + r] = v.x;
            Rt[(c + 1) * kRt + r] = v.y;
            Rt[(c + 2) * kRt + r] = v.z;
            Rt[(c + 3) * kRt + r] = v.w;
        }
    }
    const int r0 = 4 * (tid >> 5), c0 = 4 * (tid & 31);
    for (int zz = G - 2; zz >= 0; --zz) {
        {
            const float4* src = reinterpret_cast<const float4*>(seg + (int64_t)zz * 128 * 128);
            float4* dst = reinterpret_cast<float4*>(F);
#pragma unroll
            for (int e = 0; e < 128 * 32 / 256; ++e) dst[tid + 256 * e] = __ldg(src + tid + 256 * e);
        }
        __syncthreads();
        float acc[4][4];
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
            for (int c = 0; c < 4; ++c) acc[r][c] = 0.f;
#pragma unroll 8
        for (int k = 0; k < 128; ++k) {
            const float4 a = *reinterpret_cast<const float4*>(Rt + k * kRt + r0);
            const float4 f = *reinterpret_cast<const float4*>(F + k * 128 + c0);
            const float av[4] = {a.x, a.y, a.z, a.w}, fv[4] = {f.x, f.y, f.z, f.w};
#pragma unroll
            for (int r = 0; r < 4; ++r)
#pragma unroll
                for (int c = 0; c < 4; ++c) acc[r][c] = fmaf(av[r], fv[c], acc[r][c]);
        }
        __syncthreads();
        if (zz > 0) {
#pragma unroll
            for (int r = 0; r < 4; ++r)
#pragma unroll
                for (int c = 0; c < 4; ++c) Rt[(c0 + c) * kRt + r0 + r] = acc[r][c];
        } else {
            float* out = M + item * 128 * 128 + (int64_t)(kMergeRows * rb + r0) * 128 + c0;
#pragma unroll
            for (int r = 0; r < 4; ++r)
                *reinterpret_cast<float4*>(out + r * 128) = make_float4(acc[r][0], acc[r][1], acc[r][2], acc[r][3]);
        }
    }
}

}  // namespace

// Segments per M chain: at most (P - 2) * Hv chains (the first and the last
// shard never span) run two CTAs to an SM; G segments of nch / G chunks take
// ceil(chains * G / slots) rounds, and the merge adds G - 1 products per
// chain, about a tenth of a chunk period each over the whole GPU (measured:
// 0.13-0.18 us per chain and product against 1.7 us per chunk).  G > 1 only
// where that cuts the modelled time by a fifth or more, with segments of 16
// chunks at least.
int mchain_segments(int T, int P, int Hv) {
    if (P < 3 || T <= 0) return 1;
    const long long nch = ((long long)(T / P) + 63) / 64;
    const long long chains = (long long)(P - 2) * Hv, slots = 2ll * device_sm_count();
    auto cost = [&](long long G) {
        return 10 * ((chains * G + slots - 1) / slots) * ((nch + G - 1) / G) + chains * (G - 1);
    };
    long long best = 1;
    for (long long G = 2; G <= 8 && nch / G >= 16; ++G)
        if (cost(G) < cost(best)) best = G;
    return 5 * cost(best) <= 4 * cost(1) ? (int)best : 1;
}

bool mchain_eligible(gdn_dtype dt, int dk, int dv) { return dt == GDN_BF16 && dk == 128 && dv == 128; }

size_t mchain_scratch_bytes(int T, int P, int Hv) {
    if (P < 2) return 0;
    const size_t nch = ((size_t)(T / P) + 63) / 64;
    const size_t chunks = (size_t)P * Hv * nch;
    const int G = mchain_segments(T, P, Hv);
    return 2 * al256(chunks * 64 * 128 * sizeof(bf16)) + al256(chunks * sizeof(float)) +
           (G > 1 ? al256((size_t)G * P * Hv * 128 * 128 * sizeof(float)) : 0);
}

gdn_status launch_mchain(const int32_t* plan, int num_seqs, int T, int P, int Hv, void* w, void* kt,
                         const float* eg, float* M, cudaStream_t s) {
    if (P < 2 || T <= 0) return GDN_OK;
    MParams p{};
    p.plan = plan; p.num_seqs = num_seqs; p.P = P; p.Hv = Hv; p.nch = (T / P + 63) / 64;
    p.eg = eg; p.M = M;
    const int G = mchain_segments(T, P, Hv);
    // the segments' products follow e^{G_last} in the scratch
    p.Mseg = reinterpret_cast<float*>(const_cast<char*>(reinterpret_cast<const char*>(eg)) +
                                      al256((size_t)P * Hv * p.nch * sizeof(float)));
    const int64_t rows = (int64_t)P * Hv * p.nch * 64;
    MMaps maps;
    memset(&maps, 0, sizeof(maps));
    gdn_status st;
    if ((st = make_map_bf16(&maps.w, w, 128, 128, rows)) != GDN_OK) return st;
    if ((st = make_map_bf16(&maps.kt, kt, 128, 128, rows)) != GDN_OK) return st;
    // at most two CTAs to an SM, the two that its tensor memory holds (a third
    // would only wait in its allocation, keeping a place a chain could use)
    const size_t smem = sizeof(MSmem) + 1024 > kMSmemFloor ? sizeof(MSmem) + 1024 : kMSmemFloor;
    if ((st = set_smem_attr((const void*)mchain_kernel, smem)) != GDN_OK) return st;
    mchain_kernel<<<dim3(P, Hv, G), MT, smem, s>>>(p, maps);
    if ((st = check_launch("mchain_kernel")) != GDN_OK || G == 1) return st;
    if ((st = set_smem_attr((const void*)mchain_merge_kernel, kMergeSmem)) != GDN_OK) return st;
    mchain_merge_kernel<<<dim3(P * Hv, 128 / kMergeRows), 256, kMergeSmem, s>>>(plan, Hv, G, p.Mseg, M);
    return check_launch("mchain_merge_kernel");
}

}  // namespace gdn
