// bf16 chunk kernel for d_k = d_v = 128 on the 5th-generation tensor cores
// (tcgen05.mma, accumulators in tensor memory).
//
// A CTA runs jobs: a job is a token range of one value head with the full
// 128-column state, chunk after chunk (C = 64).  Every product has M = 128
// (a head dimension); the state is kept transposed, S^T [value][key], in
// tensor memory (thread = value row).  Per chunk, with the chunk's in-chunk
// gate prefix G, Q~ = diag(scale e^G / |q|) Q, K~ = diag(e^{G_last - G} / |k|) K,
// Tbg = T diag(beta e^G / |k|), Tb = T diag(beta), T = (I + L)^-1 and
// A = scale Q^ K^T o Gamma (lower, diagonal included):
//   [Q;K] K^T                   -> the Q K^T and K K^T blocks (A and L)
//   W^T = K^T Tbg^T,  U^T = V^T Tb^T
//   v_new^T = U^T - S^T W^T      the state-dependent chain, part 1
//   o^T     = S^T Q~^T           (off the chain)
//   S^T    <- e^{G_last} S^T + v_new^T K~    the chain, part 2
//   o^T    += v_new^T A^T        (off the chain)
// Only the two chain products and the tensor-memory <-> shared-memory moves
// of v_new and S are serial from chunk to chunk; everything else works a
// chunk ahead.  Operands sit in shared memory in the 128-byte-swizzled
// canonical layouts: the Q/K tiles and A K-major, K~ MN-major (a row-scaled
// copy of the K rows), and W K-major in the K rows of its Q/K tile once K~ is
// copied (read out of tensor memory one key row per thread); v_new and the
// bf16 state are A operands in tensor memory.  No operand is transposed
// element by element.
//
// Two roles of two warpgroups each work on different chunks at once:
//   producer (warps 0-7), chunk g, a chunk ahead of the consumer:
//     A) warps 1-7 read A and L out of chunk g's [rows] K^T columns (once
//        chunk g-2's output products have read the A slot); thread 0 waits
//        for chunk g-1's W/U products and issues chunk g's V load;
//     B) warps 0-3 run the UT inverse (tf32 mma.sync 16x16 blocks, written as
//        the bf16 operands Tb and Tbg), then thread 0 issues W^T and U^T
//        once V has landed and the consumer has read chunk g-1's W; beside
//        them warps 4-7 load chunk g+1's g and beta, take jobs / fill chunk
//        infos three chunks ahead, issue chunk g+1's [rows] K^T once its Q/K
//        have landed (thread 224) and take its L2 norms, gate prefix and
//        per-row factors;
//   consumer (warps 8-15), chunk g: writes the previous chunk's output
//     (staged for 16-byte stores; the gated-norm epilogue in the layer
//     instantiation), forms -Q~ in place and the K~ copy, moves W^T out of
//     tensor memory into the K rows, issues the first product, refills the
//     freed Q/K slot with chunk g+2 (TMA, 128-byte swizzle = operand layout),
//     packs v_new to bf16 in place in tensor memory (the A operand of the
//     second product), issues the second product, and while it runs forms
//     chunk g+1's -Q~ / K~ and reads its W if that chunk's W/U are done.
// A chunk whose output is not written (a summary job) uses no Q: its Q norms,
// A read-out and -Q~ are skipped, and its first product takes the W rows
// alone (N = 64, straight into v_new's columns).
// The fp32 state stays in tensor memory: after each update it is read once
// for its bf16 copy (the next chunk's A operand) and written back scaled by
// the next chunk's e^{G_last}, onto which the next update accumulates.
//
// Work: one job is a token range of one value head.  With a work queue the
// grid is one persistent CTA per SM; its chunks form one stream over the jobs
// it takes (by ticket, in the order a separate kernel has sorted), so the
// pipeline runs on across job boundaries: a job's first chunk loads its
// initial state, its last stores the final state (a split item's first half
// hands it to the second half through a release flag).  Without one, every
// CTA runs the job of its block.  Every wait is bounded: on expiry the
// kernel counts a timeout and writes GDN_ERR_TIMEOUT to the launch's status
// word, both roles leave their loops, outstanding copies and products are
// waited for (bounded), and the tensor memory is freed.
#include <cuda.h>
#include <string.h>

#include "chunk_common.cuh"
#include "tc_util.cuh"

namespace gdn {

__device__ int g_gdn_timeouts;  // bounded waits that expired (read by gdn_device_timeouts)

#ifdef GDN_PHASE_STAMPS
// Phase timestamps (clock64) of CTA 0 for chunks [kStamp0, kStamp0 + kStampN)
// of its stream, 32 slots per chunk; a profiling build only.
constexpr int kStamp0 = 24, kStampN = 32;
__device__ long long g_gdn_stamps[kStampN * 32];
#define GDN_STAMP(gq, idx)                                                           \
    do {                                                                             \
        if (blockIdx.x == 0 && (gq) >= kStamp0 && (gq) < kStamp0 + kStampN)          \
            g_gdn_stamps[((gq) - kStamp0) * 32 + (idx)] = clock64();                 \
    } while (0)
#else
#define GDN_STAMP(gq, idx) \
    do {                   \
    } while (0)
#endif

namespace {

constexpr int NT = 512;
constexpr int GS = 256;  // threads per role (two warpgroups)
constexpr int LDF = 68;
constexpr uint32_t kSpin = 1u << 20;  // try_wait polls before a wait is declared stuck
constexpr int BAR_P = 1, BAR_S = 2;   // named barriers of the two roles
constexpr int BAR_PA = 3;             // producer warps 0-3 (the UT inverse)
constexpr int BAR_Q = 4;              // producer warps 1-7 (A/L readout)
constexpr int BAR_R = 5;              // producer warps 4-7 (next chunk's factors)
typedef __nv_bfloat16 bf16;

struct TmaMaps {
    CUtensorMap q, k, v;  // [T rows x heads*128 columns] bf16 views, 64x64 boxes, 128-byte swizzle
    CUtensorMap wst, kst;  // stored W rows / K~ of spanning shards' chunks (same boxes), when the M chains run apart
};

// Per-slot values that only the producer reads (written a chunk ahead).
struct SlotSmall {
    float qf[64];    // scale e^{G_i} / |q_i|: row factor of Q~
    float fac[64];   // e^{G_last - G_j} / |k_j|: row factor of K~
    float beta[64];  // beta_j
    float fbg[64];   // beta_j e^{G_j} / |k_j|: column factor of Tbg
};

// One job of a CTA's chunk stream (shared memory).  span = {global index of
// the job's first chunk in the stream, chunks}: one 64-bit word, written
// last, so a reader scanning the ring sees either a whole old span or the
// whole new one.
struct JobRec {
    int2 span;
    int t0, t1;        // tokens [t0, t1)
    int hv, hk, col0;
    int write_o, value_zero, identity_init;
    int part, flag;    // split half (0 whole, 1 first, 2 second); hand-over flag index
    int wk_base;       // >= 0: store the chunks' W rows, K~ and e^{G_last} from this slot on
    const float* init;
    float* fin;
    int64_t init_ld, fin_ld;
};
constexpr int kRing = 8;  // jobs in flight per CTA: at most about 5 are live at once

// What the roles need of one chunk of the stream, filled three chunks ahead
// (entry gq & 7 holds chunk gq; it is overwritten when chunk gq + 8 is filled,
// by which time both roles are past chunk gq).  eglast is written by the
// producer's gate prefix of the chunk, a chunk ahead of the consumer.
struct ChunkInfo {
    int tb, valid;      // first token, valid rows
    int hv, hk;         // value head, key head
    int vz, write_o;    // value columns zero; o written
    int first, last;    // first / last chunk of its job
    int jr;             // ring entry of its job
    float eglast;       // e^{G_last}
    int eg_ready;       // == the chunk's stream index once its gate prefix and factors are written
    int aread;          // == the chunk's stream index once its [rows] K^T columns have been read
};

struct SmemWS {
    bf16 QK[2][128 * 128];  // per slot: slot 0 [K;Q], slot 1 [Q;K]; Q becomes -Q~ in place, K becomes W once read
    bf16 KT[2][64 * 128];   // per slot: K~ [token][key], MN-major B of the state update
    bf16 A[2][64 * 64];     // per slot: A [token][token], K-major B of the output update
    bf16 V[64 * 128];       // [token][value column]
    bf16 Tb[64 * 64];       // T diag(beta)
    bf16 Tbg[64 * 64];      // T diag(beta e^G / |k|)
    bf16 OST[64 * 128];     // output staging: [token][value column]
    __align__(16) float LT[64 * LDF];  // L; the inverse's blocks replace it block by block
    SlotSmall slot[2];
    __align__(16) float G[64];
    __align__(16) float eG[64];
    __align__(16) float eGl[64];
    __align__(16) float rn[128];  // 1/|q_i| (0-63), 1/|k_j| (64-127); 1 without the L2-norm flag
    // split decay mask e^{G_i - G_j} = e^{G_i - G_r} e^{G_r - G_j}, with one
    // reference token r_b = 16 b + 7 per 16-row block b of the rows i
    __align__(16) float colf[4][64];  // e^{G_{r_b} - G_j} / |k_j|
    __align__(16) float rowA[64];     // scale e^{G_i - G_r} / |q_i|
    __align__(16) float rowL[64];     // beta_i e^{G_i - G_r} / |k_i|
    float Gref[4];
    int factored;                  // the split factors stay well inside fp32 range
    uint64_t mbar_p, mbar_s, mbar_o;  // tensor-core completion: Gram; chain products; output products
    uint64_t full[2], wfree;       // chunk ready for the consumer; W columns read
    uint64_t afree[2];             // per A slot: the chunk's output products are done (A may be rewritten)
    uint64_t ld_qk[2], ld_v;       // TMA arrivals (transaction bytes)
    uint64_t fin_p, fin_s, fin_s2;  // end-of-kernel drains of the issuing threads' products
    int qk_issued[2], qk_waited[2], v_issued, v_waited;
    uint32_t tmem_slot;
    int lpt_len[kMaxLptItems];
    int lpt_pick;
    JobRec ring[kRing];
    int jn;        // jobs pushed into the ring
    int jdone;     // jobs the consumer has finished (their entries may be reused)
    int chunks;    // chunks of the pushed jobs
    int src_end;   // the job source is exhausted
    int lpt_left;  // without a work queue: the CTA's one job is still to be pushed
    int lpt_b[3];
    int acq_ok;    // the first jobs were pushed without a ring timeout
    int abort;     // a role gave up: every bounded wait of the other role returns
    ChunkInfo ci[8];
    float ored[4][64];  // gated norm: per value-lane quarter, each token's sum of o^2
};

constexpr uint32_t ID_N64 = tc::idesc_bf16(128, 64, false, false, false);
constexpr uint32_t ID_N64_AMN = tc::idesc_bf16(128, 64, true, false, false);
constexpr uint32_t ID_N128_NEG = tc::idesc_bf16(128, 128, false, false, false) | (1u << 14);  // B negated
constexpr uint32_t ID_N64_NEG = ID_N64 | (1u << 14);
constexpr uint32_t ID_N128_BMN = tc::idesc_bf16(128, 128, false, true, false);

// One warp: the chunk's gate prefix from per-token values held by lanes
// (lane l holds g of tokens 2l and 2l+1; beta likewise), written to shared
// memory with e^G, e^{G_last - G}, beta, the block references of the split
// decay mask and whether the split factors stay within fp32 range: inside a
// block b, |G_i - G_{r_b}| < 60, and G_{r_b} - G_j < 60 for every j up to the
// block's end (a column factor that underflows stands for a decay product
// that underflows as well).  e^{G_last} goes to the chunk's info entry.
template <class Sm>
__device__ __forceinline__ void gate_prefix_fast(Sm& sm, SlotSmall& sl, ChunkInfo& ci, float g0, float g1, float b0,
                                                 float b1) {
    const int lane = threadIdx.x & 31;
    float s = g0 + g1;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const float t = __shfl_up_sync(0xffffffffu, s, off);
        if (lane >= off) s += t;
    }
    const float G1 = s, G0 = s - g1;
    const float Gl = __shfl_sync(0xffffffffu, s, 31);
    const float Gr = __shfl_sync(0xffffffffu, G1, (lane & ~7) + 3);  // G of token 16 b + 7
    float mn = fminf(G0, G1);  // running minimum of G
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const float t = __shfl_up_sync(0xffffffffu, mn, off);
        if (lane >= off) mn = fminf(mn, t);
    }
    const float mend = __shfl_sync(0xffffffffu, mn, lane | 7);  // through the block's last token
    float dev = fmaxf(fmaxf(fabsf(G0 - Gr), fabsf(G1 - Gr)), Gr - mend);
#pragma unroll
    for (int off = 16; off; off >>= 1) dev = fmaxf(dev, __shfl_xor_sync(0xffffffffu, dev, off));
    sm.G[2 * lane] = G0;
    sm.G[2 * lane + 1] = G1;
    sm.eG[2 * lane] = __expf(G0);
    sm.eG[2 * lane + 1] = __expf(G1);
    sm.eGl[2 * lane] = __expf(Gl - G0);
    sm.eGl[2 * lane + 1] = __expf(Gl - G1);
    sl.beta[2 * lane] = b0;
    sl.beta[2 * lane + 1] = b1;
    if ((lane & 7) == 3) sm.Gref[lane >> 3] = Gr;
    if (lane == 0) {
        sm.factored = dev < 60.f;
        ci.eglast = __expf(Gl);
    }
}

// One warp: 32 values per lane in, lane l out with the sum over the warp's
// lanes of their value l (a butterfly that halves the values each step).
__device__ __forceinline__ float reduce_scatter32(float (&v)[32]) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int k = 16; k >= 1; k >>= 1) {
        const bool up = (lane & k) != 0;
#pragma unroll
        for (int i = 0; i < k; ++i) {
            const float send = up ? v[i] : v[i + k];
            const float keep = up ? v[i + k] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, k);
        }
    }
    return v[0];
}

// Flag hand-over between the two halves of a split item (global memory).
__device__ __forceinline__ void st_release(int32_t* p, int32_t v) {
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ int32_t ld_acquire(const int32_t* p) {
    int32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
// Waits (at most `limit_ns` of the global timer) for a released flag; false
// on expiry.
__device__ __forceinline__ bool wait_flag(const int32_t* f, long long limit_ns, const volatile int* abort) {
    uint64_t t0;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
    for (uint32_t it = 0; it < (1u << 26); ++it) {
        if (ld_acquire(f)) return true;
        if (*abort) return false;
        uint64_t t;
        asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
        if ((long long)(t - t0) > limit_ns) return false;
        __nanosleep(256);
    }
    return false;
}

__device__ __forceinline__ uint4 pack8(const float* f) {
    uint4 r;
    __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&r);
#pragma unroll
    for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
    return r;
}

// bf16 copies of -acc (a 16x16 block at block position (bi, bj) of T) into
// Tb = T diag(beta) and Tbg = T diag(fbg).
__device__ __forceinline__ void store_tb16_neg(const float (&acc)[2][4], bf16* Tb, bf16* Tbg, const float* beta,
                                               const float* fbg, int bi, int bj) {
    const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
        const int J = 16 * bj + 8 * nt + 2 * t;
        const float2 b2 = *reinterpret_cast<const float2*>(beta + J), f2 = *reinterpret_cast<const float2*>(fbg + J);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int e = tc::sw128(64, 16 * bi + g + 8 * h, J);
            const float v0 = -acc[nt][2 * h], v1 = -acc[nt][2 * h + 1];
            *reinterpret_cast<__nv_bfloat162*>(Tb + e) = __floats2bfloat162_rn(v0 * b2.x, v1 * b2.y);
            *reinterpret_cast<__nv_bfloat162*>(Tbg + e) = __floats2bfloat162_rn(v0 * f2.x, v1 * f2.y);
        }
    }
}

// Tb = T diag(beta) and Tbg = T diag(fbg) (bf16, 128-byte-swizzled K-major
// 64x64) for T = (I + L)^-1, the strictly lower L in Ls (fp32, row stride
// LDF), on 128 threads (gtid 0-127; `sync` is their barrier).  16x16 blocks:
// the diagonal blocks D_a = (I + L_aa)^-1 by forward substitution (one column
// per thread); then warps 0 and
// 1 form T10 = -D1 (L10 D0) and T32 = -D3 (L32 D2) while warps 2 and 3 start
// X = C A0^-1 for the lower-left 32x32 block C (X_a0 = L_a0 D0 + L_a1 T10,
// X_a1 = L_a1 D1) and write the bf16 copies of D0-D3; finally the lower-left
// blocks T_2b = -D2 X_2b and T_3b = -(T32 X_2b + D3 X_3b).  Block products are
// tf32 mma.sync; each result replaces the L block that only its own warp
// still reads.  Blocks above the diagonal are never written: Tb and Tbg hold
// zeros there from the start.
template <class Sync>
__device__ __forceinline__ void ut_inverse_tb(float* Ls, bf16* Tb, bf16* Tbg, const float* beta, const float* fbg,
                                              int gtid, Sync sync, int gq) {
    (void)gq;
    const int gw = gtid >> 5;
    auto blk = [&](int a, int b) { return Ls + 16 * a * LDF + 16 * b; };
    // bf16 copies of a final 16x16 block of T, 8 columns per step: t < 128 the
    // diagonal blocks D0-D3, 128-159 T10, 160-191 T32
    auto tb_copy = [&](int t) {
        const int bk = t >> 5, r = (t >> 1) & 15, h = t & 1;
        const int bi = bk < 4 ? bk : (bk == 4 ? 1 : 3), bj = bk < 4 ? bk : (bk == 4 ? 0 : 2);
        const int J = 16 * bj + 8 * h;
        const float* src = Ls + (16 * bi + r) * LDF + J;
        const float4 v0 = *reinterpret_cast<const float4*>(src), v1 = *reinterpret_cast<const float4*>(src + 4);
        const float4 b0 = *reinterpret_cast<const float4*>(beta + J), b1 = *reinterpret_cast<const float4*>(beta + J + 4);
        const float4 f0 = *reinterpret_cast<const float4*>(fbg + J), f1 = *reinterpret_cast<const float4*>(fbg + J + 4);
        const float tb[8] = {v0.x * b0.x, v0.y * b0.y, v0.z * b0.z, v0.w * b0.w,
                             v1.x * b1.x, v1.y * b1.y, v1.z * b1.z, v1.w * b1.w};
        const float tg[8] = {v0.x * f0.x, v0.y * f0.y, v0.z * f0.z, v0.w * f0.w,
                             v1.x * f1.x, v1.y * f1.y, v1.z * f1.z, v1.w * f1.w};
        const int e = tc::sw128_chunk(64, 16 * bi + r, J >> 3);
        *reinterpret_cast<uint4*>(Tb + e) = pack8(tb);
        *reinterpret_cast<uint4*>(Tbg + e) = pack8(tg);
    };
    if (gtid < 64) {
        const int da = gtid >> 4, dc = gtid & 15;
        float* Lb = blk(da, da);
        float x[16];  // column dc of D_a; rows above dc are exactly zero
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            float acc = (i == dc) ? 1.f : 0.f;
#pragma unroll
            for (int m4 = 0; m4 < i; m4 += 4) {
                const float4 l = *reinterpret_cast<const float4*>(Lb + i * LDF + m4);
                acc = fmaf(-l.x, x[m4], acc);
                if (m4 + 1 < i) acc = fmaf(-l.y, x[m4 + 1], acc);
                if (m4 + 2 < i) acc = fmaf(-l.z, x[m4 + 2], acc);
                if (m4 + 3 < i) acc = fmaf(-l.w, x[m4 + 3], acc);
            }
            x[i] = (i >= dc) ? acc : 0.f;
        }
        __syncwarp();
#pragma unroll
        for (int i = 0; i < 16; ++i) Lb[i * LDF + dc] = x[i];
    }
    sync();
    if (gtid == 0) GDN_STAMP(gq, 11);
    float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    float acc2[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    if (gw < 2) {
        const int a = gw ? 3 : 1, b = a - 1;
        mma_block16_tf32<LDF>(acc, blk(a, b), blk(b, b));
        __syncwarp();
        store_block16<LDF>(acc, blk(a, b));
        __syncwarp();
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[nt][e] = 0.f;
        mma_block16_tf32<LDF>(acc, blk(a, a), blk(a, b));
        __syncwarp();
        store_block16_neg<LDF>(acc, blk(a, b));
    } else {
        mma_block16_tf32<LDF>(acc, blk(gw, 0), blk(0, 0));
        mma_block16_tf32<LDF>(acc2, blk(gw, 1), blk(1, 1));
        tb_copy(gtid - 64);
        tb_copy(gtid);
    }
    sync();
    if (gtid == 0) GDN_STAMP(gq, 12);
    if (gw >= 2) {
        mma_block16_tf32<LDF>(acc, blk(gw, 1), blk(1, 0));
        __syncwarp();
        store_block16<LDF>(acc, blk(gw, 0));
        store_block16<LDF>(acc2, blk(gw, 1));
    } else {
        tb_copy(128 + gtid);  // T10 and T32 are final
    }
    sync();
    if (gtid == 0) GDN_STAMP(gq, 13);
    {
        const int a = 2 + (gw >> 1), b = gw & 1;
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[nt][e] = 0.f;
        if (a == 2) {
            mma_block16_tf32<LDF>(acc, blk(2, 2), blk(2, b));
        } else {
            mma_block16_tf32<LDF>(acc, blk(3, 2), blk(2, b));
            mma_block16_tf32<LDF>(acc, blk(3, 3), blk(3, b));
        }
        store_tb16_neg(acc, Tb, Tbg, beta, fbg, a, b);
    }
}

// One thread: pushes jobs into the CTA's ring until the stream holds at
// least `need` chunks or the source is exhausted.  With a work queue a job is
// the entry of the next ticket (whole item or half, for one (head, tile)
// pair); without one, the CTA's own block.  Jobs without work are skipped;
// with a work queue so are jobs without tokens (their final states are
// written by a separate kernel).  False when the ring stayed full (a bounded
// wait for the consumer expired).
__device__ __noinline__ bool acquire_jobs(const ChunkParams& p, int src, SmemWS& sm, int need) {
    volatile int* vdone = &sm.jdone;
    while (!sm.src_end && sm.chunks < need) {
        if (sm.jn - *vdone >= kRing) {
            const volatile int* vab = &sm.abort;
            for (uint32_t it = 0; it < kSpin && sm.jn - *vdone >= kRing && !*vab; ++it) __nanosleep(64);
            if (sm.jn - *vdone >= kRing) return false;
        }
        int bx, by, bz, part = 0, first_chunks = 0, flag = 0;
        if (p.sched) {
            const int m = p.sched_m;
            const int t = atomicAdd(p.sched, 1);
            const int r = t / m, rem = t - r * m;
            if (r >= __ldcg(p.sched + 1)) {
                sm.src_end = 1;
                break;
            }
            const int2 ent =
                __ldcg(reinterpret_cast<const int2*>(p.sched + chunk_sched_order_off(p.sched_items, m)) + r);
            bx = ent.x & 0xffff;
            part = ent.x >> 16;
            first_chunks = ent.y;
            by = rem % p.sched_ny;
            bz = rem / p.sched_ny;
            flag = bx * m + rem;
        } else {
            if (!sm.lpt_left) {
                sm.src_end = 1;
                break;
            }
            sm.lpt_left = 0;
            bx = sm.lpt_b[0];
            by = sm.lpt_b[1];
            bz = sm.lpt_b[2];
        }
        ChunkJob job;
        if (!make_job(p, src, job, bx, by, bz)) continue;
        if (part) {  // a part of a split item, handed over through a final-state destination
            // a continuing pass-2 segment has none of its own: its start state
            // (read once, by the first part) takes the first part's final state
            float* hand = job.fin;
            int64_t hand_ld = job.fin_ld;
            if (!hand && src == JOBS_SHARD_PASS2) {
                hand = const_cast<float*>(job.init);
                hand_ld = job.init_ld;
            }
            if (!hand) {  // nowhere to hand over: the first part runs the whole item
                if (part == 2) continue;
                part = 0;
            } else {
                const int split_t = job.t0 + 64 * first_chunks;
                if (part == 1) {
                    job.t1 = split_t;
                    job.fin = hand;
                    job.fin_ld = hand_ld;
                } else {
                    job.t0 = split_t;
                    job.init = hand;
                    job.init_ld = hand_ld;
                    job.identity_init = false;  // an M summary continues from its first part's M
                    if (job.wk_base >= 0) job.wk_base += first_chunks;  // stored operands: chunk slots
                }
            }
        }
        const int nch = (job.t1 - job.t0 + 63) / 64;
        if (nch == 0 && p.sched) continue;
        JobRec& J = sm.ring[sm.jn % kRing];
        J.t0 = job.t0;
        J.t1 = job.t1;
        J.hv = job.hv;
        J.hk = job.hv / (p.Hv / p.Hk);
        J.col0 = job.col0;
        J.write_o = job.write_o;
        J.value_zero = job.value_zero;
        J.identity_init = job.identity_init;
        J.part = part;
        J.flag = flag;
        J.init = job.init;
        J.fin = job.fin;
        J.init_ld = job.init_ld;
        J.fin_ld = job.fin_ld;
        J.wk_base = job.wk_base;
        __threadfence_block();
        *reinterpret_cast<volatile unsigned long long*>(&J.span) =
            ((unsigned long long)(unsigned)nch << 32) | (unsigned)sm.chunks;  // {first chunk, chunks}
        __threadfence_block();
        sm.chunks += nch;
        sm.jn += 1;
    }
    return true;
}

// One thread: the info of chunk gq (already in the stream) from its job.
__device__ __forceinline__ void fill_chunk_info(SmemWS& sm, int gq) {
    int r = 0;
#pragma unroll
    for (int i = 0; i < kRing; ++i) {
        const int2 sp = sm.ring[i].span;
        if (gq >= sp.x && gq < sp.x + sp.y) r = i;
    }
    const JobRec& J = sm.ring[r];
    const int c = gq - J.span.x;
    ChunkInfo& I = sm.ci[gq & 7];
    I.tb = J.t0 + 64 * c;
    I.valid = min(64, J.t1 - I.tb);
    I.hv = J.hv;
    I.hk = J.hk;
    I.vz = J.value_zero;
    I.write_o = J.write_o;
    I.first = c == 0;
    I.last = c == J.span.y - 1;
    I.jr = r;
}

// With a work queue, sequences without tokens are not queued: the persistent
// CTAs share them out and write their final states (h0, or 0), all threads.
__device__ __forceinline__ void empty_sequences_final(const ChunkParams& p, int src) {
    if (!p.sched || src != JOBS_SEQS || !p.h_final) return;
    const int64_t sz = (int64_t)p.Hv * p.dk * p.dv;
    for (int n = blockIdx.x; n < p.num_seqs; n += gridDim.x) {
        if (__ldg(p.cu + n) != __ldg(p.cu + n + 1)) continue;
        float* hf = p.h_final + n * sz;
        const float* h0 = p.h0 ? p.h0 + n * sz : nullptr;
        for (int64_t e = threadIdx.x; e < sz; e += NT) hf[e] = h0 ? h0[e] : 0.f;
    }
}


// ---- helpers of the kernel (each is called from more than one place) ----

// Q/K of chunk gq into its slot: four 64x64 boxes (128-byte swizzle = the
// operand layout); slot 0 holds [K;Q], slot 1 [Q;K]; one thread
__device__ __forceinline__ void issue_qk_fn(SmemWS& sm, const TmaMaps& maps, const ChunkParams& p, int gq, int tbn,
                                         int hk) {
    const int ss = gq & 1;
    bf16* qd = sm.QK[ss] + (ss ? 0 : 64 * 64);
    bf16* kd = sm.QK[ss] + (ss ? 64 * 64 : 0);
    uint64_t* bar = &sm.ld_qk[ss];
    // token-major views [T x Hk*128]: (hk*128 + c, t); head-major [Hk*T x 128]: (c, hk*T + t)
    const int x0 = p.head_major ? 0 : hk * 128, y0 = p.head_major ? hk * p.T + tbn : tbn;
    tc::mbar_expect_tx(bar, 4 * 64 * 64 * 2);
    tc::tma_load_2d(qd, &maps.q, x0, y0, bar);
    tc::tma_load_2d(qd + 128 * 64, &maps.q, x0 + 64, y0, bar);
    tc::tma_load_2d(kd, &maps.k, x0, y0, bar);
    tc::tma_load_2d(kd + 128 * 64, &maps.k, x0 + 64, y0, bar);
    sm.qk_issued[ss] += 1;
}

// V of chunk gq (unless its value columns are zero); one thread
__device__ __forceinline__ void issue_v_fn(SmemWS& sm, const TmaMaps& maps, const ChunkParams& p, int gq) {
    const ChunkInfo& I = sm.ci[gq & 7];
    if (!I.vz) {
        const int tbn = I.tb, hv = I.hv;
        const int x0 = p.head_major ? 0 : hv * 128, y0 = p.head_major ? hv * p.T + tbn : tbn;
        tc::mbar_expect_tx(&sm.ld_v, 2 * 64 * 64 * 2);
        tc::tma_load_2d(sm.V, &maps.v, x0, y0, &sm.ld_v);
        tc::tma_load_2d(sm.V + 64 * 64, &maps.v, x0 + 64, y0, &sm.ld_v);
        sm.v_issued += 1;
    }
}

// [rows] K^T of chunk gq once its Q/K have landed (one thread; dA = the
// slot's 128 rows, dB = its K rows); true when the load arrived
__device__ __forceinline__ bool issue_gram_fn(SmemWS& sm, uint32_t t_gram, uint64_t dA, uint64_t dB, int gq) {
    const int ss = gq & 1;
    if (!tc::mbar_wait(&sm.ld_qk[ss], (gq >> 1) & 1, kSpin, &sm.abort)) return false;
    sm.qk_waited[ss] += 1;
    tc::fence_after();
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) tc::mma(t_gram, dA + tc::koff(128, kk), dB + tc::koff(128, kk), ID_N64, kk > 0);
    tc::commit(&sm.mbar_p);
    return true;
}

// warps 4-7 (one row each, r = gt - 128): the L2 norms of chunk gq's rows
// (rn[0-63] Q rows, rn[64-127] K rows); one thread waits for the load
__device__ __forceinline__ bool norms_fn(SmemWS& sm, int gq, int gt, bool l2) {
    const int ss = gq & 1;
    bool in = true;
    if (gt == 128) in = tc::mbar_wait(&sm.ld_qk[ss], (gq >> 1) & 1, kSpin, &sm.abort);
    if (!tc::bar_and(BAR_R, 128, in)) return false;
    if (gt == 128) GDN_STAMP(gq - 1, 14);
    const int r = gt - 128;
    float acc0 = 0.f, acc1 = 0.f;
    const bool qskip = (ss ? (r < 64) : (r >= 64)) && !sm.ci[gq & 7].write_o;  // no output: Q norms unused
    if (l2 && !qskip) {
        const bf16* QKn = sm.QK[ss];
#pragma unroll 4
        for (int ch = 0; ch < 16; ++ch) {
            const uint4 raw = *reinterpret_cast<const uint4*>(&QKn[tc::sw128_chunk(128, r, ch)]);
            const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&raw);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float2 f = __bfloat1622float2(h2[i]);
                acc0 = fmaf(f.x, f.x, acc0);
                acc1 = fmaf(f.y, f.y, acc1);
            }
        }
    }
    const bool qrow = ss ? (r < 64) : (r >= 64);
    sm.rn[(qrow ? 0 : 64) + (r & 63)] = l2 ? rsqrtf(acc0 + acc1 + 1e-6f) : 1.f;
    return true;
}

// warps 4-7: chunk gq's gate prefix (warp 5, from its g / beta registers)
// and per-row factors (its norms are in rn); `in` is this thread's verdict
// so far.  Publishes e^{G_last} in the chunk's info entry for the consumer.
__device__ __forceinline__ bool prep_fn(SmemWS& sm, float scale, int gq, bool in, int gt, float g0, float g1, float b0,
                                     float b1) {
    const int ss = gq & 1, warp = gt >> 5, lane = gt & 31;
    SlotSmall& sl = sm.slot[ss];
    (void)lane;
    if (warp == 5) gate_prefix_fast(sm, sl, sm.ci[gq & 7], g0, g1, b0, b1);
    if (!tc::bar_and(BAR_R, 128, in)) return false;
    if (gt == 128) GDN_STAMP(gq - 1, 15);
    const int f = gt - 128;
    if (f < 64) {
        const int i = f;
        const float r = sm.rn[i], Gi = sm.G[i];
        sm.rowA[i] = scale * r * __expf(Gi - sm.Gref[i >> 4]);
        sl.qf[i] = scale * sm.eG[i] * r;
    } else {
        const int j = f - 64;
        const float rk = sm.rn[64 + j], Gj = sm.G[j], bj = sl.beta[j];
        sm.rowL[j] = bj * rk * __expf(Gj - sm.Gref[j >> 4]);
        sl.fbg[j] = bj * sm.eG[j] * rk;
        sl.fac[j] = sm.eGl[j] * rk;
#pragma unroll
        for (int b = 0; b < 4; ++b) sm.colf[b][j] = (j < 16 * (b + 1)) ? rk * __expf(sm.Gref[b] - Gj) : 0.f;
    }
    tc::bar_sync(BAR_R, 128);  // every factor written: publish them with e^{G_last}
    if (gt == 128) {
        __threadfence_block();
        *reinterpret_cast<volatile int*>(&sm.ci[gq & 7].eg_ready) = gq;
    }
    return true;
}

// A job's initial state: its bf16 copy into the bf16 state columns (the A
// operand of the first product), and the state scaled by e^{G_last} of the
// job's first chunk (its update accumulates onto it) into the state columns.
// Thread (row, half): S^T row `row`, keys [64 half, 64 half + 64).
__device__ __forceinline__ void load_state_fn(const JobRec& J, float eg, uint32_t t_s, uint32_t t_sb, int row, int half) {
    const float* ini = J.init;
    const int64_t ild = J.init_ld;
    const bool idi = J.identity_init != 0;
    const int col0 = J.col0;
#pragma unroll 1
    for (int q4 = 0; q4 < 4; ++q4) {
        float v[16];
        uint32_t w[8];
#pragma unroll
        for (int c2 = 0; c2 < 16; ++c2) {
            const int d = 64 * half + 16 * q4 + c2;
            float s0 = 0.f;
            if (idi) s0 = (d == col0 + row) ? 1.f : 0.f;
            else if (ini) s0 = ini[(int64_t)d * ild + row];
            v[c2] = s0;
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) w[j] = tc::pack_bf16x2(v[2 * j], v[2 * j + 1]);
        tc::stw8(t_sb + 32 * half + 8 * q4, w);
#pragma unroll
        for (int c2 = 0; c2 < 16; ++c2) v[c2] *= eg;
        tc::st16(t_s + 64 * half + 16 * q4, v);
    }
}

// the job's final state from the state columns (t_s includes the lane base)
__device__ __forceinline__ void store_state_fn(const JobRec& J, uint32_t t_s, int row, int half) {
    float* fin = J.fin;
    const int64_t fld = J.fin_ld;
    if (fin) {
#pragma unroll 1
        for (int q4 = 0; q4 < 4; ++q4) {
            float v[16];
            tc::ld16(t_s + 64 * half + 16 * q4, v);
#pragma unroll
            for (int c2 = 0; c2 < 16; ++c2) fin[(int64_t)(64 * half + 16 * q4 + c2) * fld + row] = v[c2];
        }
    }
}

// W of the chunk in slot ss from tensor memory (W^T: lane = key) into the
// slot's K rows, free once K~ is copied and the W/U products have run: W
// [token][key] K-major, the first product's B rows (t_w includes the lane base)
__device__ __forceinline__ void w_readout_fn(SmemWS& sm, int ss, uint32_t t_w, int row, int half) {
    const int d = row, wrow0 = ss ? 64 : 0;
    const int dch = (d & 63) >> 3;
#pragma unroll 1
    for (int h16 = 0; h16 < 2; ++h16) {
        float wv[16];
        tc::ld16(t_w + 32 * half + 16 * h16, wv);
        bf16* wb = sm.QK[ss] + (d >> 6) * 128 * 64 + (wrow0 + 32 * half + 16 * h16) * 64 + (d & 7);
#pragma unroll
        for (int c2 = 0; c2 < 16; ++c2) wb[64 * c2 + ((dch ^ (c2 & 7)) << 3)] = __float2bfloat16_rn(wv[c2]);
    }
}

// The consumer's 256 threads (c = gt): -Q~ = -diag(qf) Q in place and
// K~ = diag(fac) K into the slot's K~ tile (same swizzled chunk positions),
// 8 chunks each, loads first so that they overlap.  Needs the chunk's
// factors (published with eg_ready) and its [rows] K^T read (aread).
__device__ __forceinline__ void qk_prep_fn(SmemWS& sm, int gq, int c) {
    const int isk0 = sm.ci[gq & 7].write_o ? 0 : 1;  // no output: K~ alone
    const int ss = gq & 1;
    const SlotSmall& sl = sm.slot[ss];
    bf16* QKs = sm.QK[ss];
    bf16* KTs = sm.KT[ss];
    const int qrow0 = ss ? 0 : 64, krow0 = 64 - qrow0;
    // the Q rows, then the K rows (kept rolled: code size); loads first
#pragma unroll 1
    for (int isk = isk0; isk < 2; ++isk) {
        const int rowb = isk ? krow0 : qrow0;
        uint4 raw[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {  // chunk e = c + 256 k
            const int e = c + 256 * k, r = e >> 4, ch = e & 15;
            raw[k] = *reinterpret_cast<const uint4*>(&QKs[tc::sw128_chunk(128, rowb + r, ch)]);
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int e = c + 256 * k, r = e >> 4, ch = e & 15;
            const float fs = isk ? sl.fac[r] : -sl.qf[r];
            const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&raw[k]);
            float x[8];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float2 t2 = __bfloat1622float2(h[i]);
                x[2 * i] = t2.x * fs;
                x[2 * i + 1] = t2.y * fs;
            }
            bf16* dst = isk ? &KTs[tc::sw128_chunk(64, r, ch)] : &QKs[tc::sw128_chunk(128, qrow0 + r, ch)];
            *reinterpret_cast<uint4*>(dst) = pack8(x);
        }
    }
}

// GNORM: the gated RMS norm output epilogue (the layer entry point); WKST:
// summary jobs may store their chunks' W rows, K~ and e^{G_last} for the M
// chains run apart (shard pass 1).  Separate instantiations, so that the plain
// forward keeps its registers and code layout.
template <bool GNORM, bool WKST>
__global__ void __launch_bounds__(NT, 1) chunk_tc_kernel(const ChunkParams p, const int src,
                                                        const __grid_constant__ TmaMaps maps) {
    extern __shared__ unsigned char smem_raw[];
    SmemWS& sm = *reinterpret_cast<SmemWS*>(smem_raw + ((1024 - (tc::smem_addr(smem_raw) & 1023)) & 1023));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    {
        int bx = blockIdx.x, by = blockIdx.y, bz = blockIdx.z;
        if (!p.sched) lpt_block<NT>(p, src, sm.lpt_len, &sm.lpt_pick, bx, by, bz);
        if (tid == 0) {
            for (int i = 0; i < kRing; ++i) sm.ring[i].span = make_int2(-1, 0);
            for (int i = 0; i < 8; ++i) sm.ci[i].eg_ready = sm.ci[i].aread = -1;
            sm.jn = sm.jdone = sm.chunks = sm.src_end = sm.abort = 0;
            sm.lpt_left = p.sched ? 0 : 1;
            sm.lpt_b[0] = bx;
            sm.lpt_b[1] = by;
            sm.lpt_b[2] = bz;
            sm.acq_ok = acquire_jobs(p, src, sm, 3) ? 1 : 0;  // the first chunks of the stream
            for (int gq = 0; gq < 3 && gq < sm.chunks; ++gq) fill_chunk_info(sm, gq);
        }
        __syncthreads();
        if (sm.jn == 0) {  // no work for this CTA
            empty_sequences_final(p, src);
            return;
        }
    }

    const bool producer = warp < 8;
    const int gt = tid & (GS - 1);  // thread index in its role
    const int row = gt & 127;       // tensor-memory lane = row of every [128 x N] product
    const int half = gt >> 7;       // which half of the columns this thread handles
    const uint32_t lb = (uint32_t)((warp & 3) * 32) << 16;

    if (tid == 0) {
        tc::mbar_init(&sm.mbar_p, 1);
        tc::mbar_init(&sm.mbar_s, 1);
        tc::mbar_init(&sm.mbar_o, 1);
        tc::mbar_init(&sm.full[0], 2);  // the W/U products' commit and a producer thread
        tc::mbar_init(&sm.full[1], 2);
        tc::mbar_init(&sm.wfree, 1);
        tc::mbar_init(&sm.afree[0], 1);
        tc::mbar_init(&sm.afree[1], 1);
        tc::mbar_init(&sm.ld_qk[0], 1);
        tc::mbar_init(&sm.ld_qk[1], 1);
        tc::mbar_init(&sm.ld_v, 1);
        tc::mbar_init(&sm.fin_p, 1);
        tc::mbar_init(&sm.fin_s, 1);
        tc::mbar_init(&sm.fin_s2, 1);
        sm.qk_issued[0] = sm.qk_issued[1] = sm.qk_waited[0] = sm.qk_waited[1] = 0;
        sm.v_issued = sm.v_waited = 0;
    }
    // A above its diagonal and the upper blocks of Tb/Tbg stay zero; the
    // readout below writes only blocks that hold kept entries
    for (int e = tid; e < 2 * 64 * 64 / 8; e += NT) reinterpret_cast<uint4*>(sm.A)[e] = make_uint4(0u, 0u, 0u, 0u);
    for (int e = tid; e < 64 * 64 / 8; e += NT) {
        reinterpret_cast<uint4*>(sm.Tb)[e] = make_uint4(0u, 0u, 0u, 0u);
        reinterpret_cast<uint4*>(sm.Tbg)[e] = make_uint4(0u, 0u, 0u, 0u);
    }
    tc::fence_async_smem();
    if (warp == 0) tc::tmem_alloc(&sm.tmem_slot, 512);
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tmem = sm.tmem_slot;
    // tensor-memory columns: [Q;K] K^T | W^T | v_new (slot 0) | o | v_new (slot 1) | S^T bf16 | S^T fp32;
    // the first product of slot 0 writes [v_new | o] = cols 128-255, of slot 1 [o | v_new] = 192-319
    const uint32_t T_GRAM = tmem, T_W = tmem + 64, T_VN0 = tmem + 128, T_O = tmem + 192, T_VN1 = tmem + 256,
                   T_SB = tmem + 320, T_S = tmem + 384;
    const uint32_t aQK0 = tc::smem_addr(sm.QK[0]), aKT0 = tc::smem_addr(sm.KT[0]), aA0 = tc::smem_addr(sm.A[0]);
    const uint32_t aV = tc::smem_addr(sm.V), aTb = tc::smem_addr(sm.Tb), aTbg = tc::smem_addr(sm.Tbg);
    bool ok = sm.acq_ok != 0;
    // base descriptors of slot 0; a K step or the other slot adds a constant
    // to the start-address field (slot 1 lies a fixed distance further on)
    constexpr uint64_t kQKslot = sizeof(bf16) * 128 * 128 / 16, kKTslot = sizeof(bf16) * 64 * 128 / 16,
                       kAslot = sizeof(bf16) * 64 * 64 / 16, kHalfRows = 64 * 128 / 16;
    const uint64_t dQK0 = tc::desc(aQK0, 16, 1024);              // the slot's 128 rows, K-major
    const uint64_t dKmn0 = tc::desc(aQK0, 128 * 128, 1024);      // K rows (slot 0: 0-63) as the MN-major A of W^T
    const uint64_t dKT0 = tc::desc(aKT0, 64 * 128, 1024);        // K~ [token][key], MN-major B
    const uint64_t dA0 = tc::desc(aA0, 16, 1024);
    const uint64_t dVmn = tc::desc(aV, 64 * 128, 1024), dTb = tc::desc(aTb, 16, 1024), dTbg = tc::desc(aTbg, 16, 1024);
    // K rows of slot ss: rows 0-63 in slot 0, 64-127 in slot 1 (Q rows the other half)
    auto krows = [&](int ss) -> uint64_t { return ss ? kQKslot + kHalfRows : 0; };

    // The CTA's chunks form one stream over its jobs, indexed by gq; every
    // barrier phase and slot follows gq.  Chunk gq is in the stream once
    // gq < chunks; the producer keeps the stream (and the chunk infos) three
    // chunks ahead of the chunk it works on.
    auto stream_len = [&]() -> int { return *reinterpret_cast<volatile int*>(&sm.chunks); };

    auto issue_qk = [&](int gq, int tbn, int hk) { issue_qk_fn(sm, maps, p, gq, tbn, hk); };
    auto issue_gram = [&](int gq) -> bool {
        const int ss = gq & 1;
        return issue_gram_fn(sm, T_GRAM, dQK0 + (ss ? kQKslot : 0), dQK0 + krows(ss), gq);
    };

    if (producer) {
        // ====================== producer warpgroups ======================
        const bool l2 = (p.flags & GDN_QK_L2NORM) != 0;
        uint32_t ph = 0;  // phase of the [rows] K^T completions
        int nvw = 0;      // thread 0: V loads waited for
        // g and beta of chunk gq into warp 5's registers (lane l: tokens 2l, 2l+1)
        float g_next0 = 0.f, g_next1 = 0.f, b_next0 = 0.f, b_next1 = 0.f;
        auto load_gb = [&](int gq) {
            if (warp == 5) {
                const ChunkInfo& I = sm.ci[gq & 7];
                const int tbn = I.tb, hv = I.hv, vn = I.valid;
                const int r0 = 2 * lane, r1 = 2 * lane + 1;
                const int64_t t0 = tbn + r0, t1 = tbn + r1;
                g_next0 = g_next1 = b_next0 = b_next1 = 0.f;
                if (r0 < vn) gate_beta<bf16>(p, t0, hv, g_next0, b_next0);
                if (r1 < vn) gate_beta<bf16>(p, t1, hv, g_next1, b_next1);
            }
        };
        auto issue_v = [&](int gq) { issue_v_fn(sm, maps, p, gq); };
        auto norms = [&](int gq) -> bool { return norms_fn(sm, gq, gt, l2); };
        auto prep = [&](int gq, bool in) -> bool {
            return prep_fn(sm, p.scale, gq, in, gt, g_next0, g_next1, b_next0, b_next1);
        };
        // A (Q rows) and L (K rows) from the [rows] K^T columns: this thread's
        // lane, columns [32 hh, 32 hh + 32)
        auto al_readout = [&](int s, int hh) {
            const bool isq = s ? (row < 64) : (row >= 64);
            const int i = row & 63;
            const int lim = isq ? i : i - 1;  // A keeps the diagonal, L does not
            // 8 columns at a time (kept rolled: code size costs instruction-fetch stalls)
#pragma unroll 1
            for (int c8 = 0; c8 < 4; ++c8) {
                const int cb = 32 * hh + 8 * c8;
                float gv[8], a[8];
                tc::ld8(T_GRAM + lb + cb, gv);
                if (sm.factored) {
                    const float fi = isq ? sm.rowA[i] : sm.rowL[i];
                    const float4* cf = reinterpret_cast<const float4*>(sm.colf[i >> 4] + cb);
                    const float4 f0 = cf[0], f1 = cf[1];
                    const float fc[8] = {f0.x, f0.y, f0.z, f0.w, f1.x, f1.y, f1.z, f1.w};
#pragma unroll
                    for (int e = 0; e < 8; ++e) a[e] = (cb + e <= lim) ? fi * (fc[e] * gv[e]) : 0.f;
                } else {  // wide gate range: one exponential per element
                    const float Gi = sm.G[i];
                    const float fi = isq ? p.scale * sm.rn[i] : sm.slot[s].beta[i] * sm.rn[64 + i];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const int j = cb + e;
                        a[e] = (j <= lim) ? fi * sm.rn[64 + j] * gv[e] * __expf(Gi - sm.G[j]) : 0.f;
                    }
                }
                if (isq) {
                    *reinterpret_cast<uint4*>(&sm.A[s][tc::sw128_chunk(64, i, cb >> 3)]) = pack8(a);
                } else {
                    float4* Lrow = reinterpret_cast<float4*>(sm.LT + i * LDF + cb);
                    Lrow[0] = make_float4(a[0], a[1], a[2], a[3]);
                    Lrow[1] = make_float4(a[4], a[5], a[6], a[7]);
                }
            }
        };
        bool pend = true;  // this thread's verdict on work whose barrier is still ahead
        if (stream_len() > 0 && ok) {
            if (gt == 32) {
                issue_qk(0, sm.ci[0].tb, sm.ci[0].hk);
                if (stream_len() > 1) issue_qk(1, sm.ci[1].tb, sm.ci[1].hk);
                issue_v(0);
            }
            if (gt >= 128) {
                load_gb(0);
                bool in = norms(0);
                if (gt == 224 && in) in = issue_gram(0);
                pend = prep(0, in);
            }
        }
        int len = stream_len();  // chunks in the stream as of the last top-up (or all of them)
        for (int g = 0; g < len && ok; ++g) {
            const int s = g & 1;
            const bool vz = gt == 0 && sm.ci[g & 7].vz != 0;  // thread 0: no U product for this chunk
            // ---- A: chunk g's [rows] K^T, then A and L (warps 1-7: warp w takes
            // lane quarter w & 3 and column half w >> 2; a half with no kept
            // entry is skipped, and warp 4 takes warp 0's quarter); thread 0
            // meanwhile waits for the previous chunk's W and U, which must have
            // read Tb, Tbg and V before the inverse and the next V load rewrite them
            if (warp != 0) {
                if (gt == 32) GDN_STAMP(g, 0);
                bool a = pend;
                if (gt == 32) a = a && tc::mbar_wait(&sm.mbar_p, ph, kSpin, &sm.abort);
                // A of chunk g replaces that of chunk g - 2 in its slot: that chunk's
                // output products must have read it
                if (gt == 32 && g >= 2) a = a && tc::mbar_wait(&sm.afree[s], ((g >> 1) - 1) & 1, kSpin, &sm.abort);
                a = tc::bar_and(BAR_Q, GS - 32, a);
                tc::fence_after();
                if (gt == 32) GDN_STAMP(g, 1);
                if (a) {
                    const int qd = warp & 3, hh = warp == 4 ? 0 : (warp >> 2);
                    const bool qq = s ? (qd < 2) : (qd >= 2);  // this warp's lanes are Q rows
                    if (!(hh == 1 && (qd & 1) == 0) && (!qq || sm.ci[g & 7].write_o)) al_readout(s, hh);  // quarters 0, 2: rows 0-31 of A / L
                }
                tc::fence_before();
                pend = tc::bar_and(BAR_Q, GS - 32, a);
                if (gt == 32) {
                    GDN_STAMP(g, 2);
                    *reinterpret_cast<volatile int*>(&sm.ci[g & 7].aread) = g;  // the Q rows may be scaled now
                }
            } else if (gt == 0 && g >= 1) {
                pend = pend && tc::mbar_wait(&sm.full[s ^ 1], ((g - 1) >> 1) & 1, kSpin, &sm.abort);
                if (pend) issue_v(g);
            }
            ph ^= 1u;
            tc::fence_async_smem();
            tc::fence_before();
            if (!(ok = tc::bar_and(BAR_P, GS, pend))) break;
            tc::fence_after();
            if (gt == 0) GDN_STAMP(g, 3);
            // ---- B: the UT inverse (warps 0-3, straight into Tb and Tbg), then
            // W/U; warps 4-7: the next chunk's g / beta, (thread 128) the stream
            // three chunks ahead (the consumer reads chunk g + 2's info once
            // chunk g's W/U are done), and the next chunk's Gram and factors
            bool nok = true;
            if (gt < 128) {
                ut_inverse_tb(sm.LT, sm.Tb, sm.Tbg, sm.slot[s].beta, sm.slot[s].fbg, gt,
                              [] { tc::bar_sync(BAR_PA, 128); }, g);
                if (gt == 0) GDN_STAMP(g, 4);
                // thread 0: W^T = K^T Tbg^T, U^T = V^T Tb^T as soon as the inverse
                // is written, once V has landed and the consumer has read the previous W
                tc::fence_async_smem();
                tc::bar_sync(BAR_PA, 128);
                if (gt == 0) {
                    bool w = true;
                    if (!vz) {
                        w = tc::mbar_wait(&sm.ld_v, nvw & 1, kSpin, &sm.abort);
                        nvw += 1;
                    }
                    if (w && g >= 1) w = tc::mbar_wait(&sm.wfree, (g - 1) & 1, kSpin, &sm.abort);
                    GDN_STAMP(g, 9);
                    if (w) {
                        if (!vz) sm.v_waited += 1;
                        tc::fence_after();
                        const uint32_t T_U = s ? T_VN1 : T_VN0;
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk) {
                            tc::mma(T_W, dKmn0 + krows(s) + tc::mnoff(kk), dTbg + tc::koff(64, kk), ID_N64_AMN, kk > 0);
                            if (!vz) tc::mma(T_U, dVmn + tc::mnoff(kk), dTb + tc::koff(64, kk), ID_N64_AMN, kk > 0);
                        }
                        tc::commit(&sm.full[s]);
                        tc::mbar_arrive(&sm.full[s]);
                    }
                    GDN_STAMP(g, 10);
                    pend = w;
                }
            } else {
                if (g + 1 < len) load_gb(g + 1);
                if (gt == 128) {
                    GDN_STAMP(g, 5);
                    // the job of chunk g + 3, taken no earlier than the pipeline needs
                    // it (the consumer loads chunk g + 2's Q/K as soon as chunk g's
                    // W/U are done, which may be before this role's next barrier; out
                    // of line, once per job), and that chunk's info
                    if (!sm.src_end && sm.chunks < g + 4) nok = acquire_jobs(p, src, sm, g + 4);
                    if (g + 3 < sm.chunks) fill_chunk_info(sm, g + 3);
                }
                if (g + 1 < len) {
                    // beside the inverse: the next chunk's [rows] K^T once its Q/K
                    // have landed (this role has read this chunk's columns), its
                    // norms, gate prefix and factors
                    if (gt == 224) nok = issue_gram(g + 1);
                    bool in = norms(g + 1);
                    if (gt == 128) GDN_STAMP(g, 6);
                    in = prep(g + 1, in);
                    if (gt == 128) GDN_STAMP(g, 7);
                    nok = nok && in;
                }
            }
            tc::fence_async_smem();
            if (!(ok = tc::bar_and(BAR_P, GS, nok))) break;
            len = stream_len();
            if (gt == 0) GDN_STAMP(g, 8);
        }
        if (ok && !pend) ok = false;  // thread 0's last W/U issue (the consumer times out as well)
        if (!ok && gt == 0) *reinterpret_cast<volatile int*>(&sm.abort) = 1;
        if (gt == 0 || gt == 224) {  // every product these threads issued has completed
            uint64_t* fb = gt == 0 ? &sm.fin_p : &sm.fin_s2;
            tc::commit(fb);
            tc::mbar_wait(fb, 0, kSpin);
        }
    } else {
        // ====================== consumer warpgroups ======================
        bf16* __restrict__ o = static_cast<bf16*>(p.o);
        uint32_t ph = 0;  // phase of the chain products' completions
        auto wait_s = [&]() -> bool {
            bool done = true;
            if (gt == 0) done = tc::mbar_wait(&sm.mbar_s, ph, kSpin, &sm.abort);
            ph ^= 1u;
            const bool all = tc::bar_and(BAR_S, GS, done);
            tc::fence_after();
            return all;
        };
        // The fp32 state lives in the state columns of tensor memory: thread
        // (row, half) holds S^T row `row` (value column), key columns
        // [64 half, 64 half + 64).  Its bf16 copy, the A operand of the first
        // product, sits in the bf16 state columns (two keys per column).
        auto load_state = [&](const JobRec& J, float eg) { load_state_fn(J, eg, T_S + lb, T_SB + lb, row, half); };
        auto store_state = [&](const JobRec& J) { store_state_fn(J, T_S + lb, row, half); };
        auto w_readout = [&](int ss) { w_readout_fn(sm, ss, T_W + lb, row, half); };
        // The output of a chunk, tensor memory -> global memory: thread (row,
        // half) holds value column `row` of tokens [32 half, 32 half + 32); a
        // warp's 32 lanes store 64 contiguous bytes of a token row at a time.
        // With the gated norm (the wrappers' norm(o, z) on rows of head_v_dim)
        // each token's sum of squares of its bf16 outputs is reduced over the
        // 128 value lanes (warp butterfly, then the four lane quarters through
        // shared memory) and the stores write norm_w * o / sqrt(mean(o^2) + eps) * silu(z).
        constexpr bool gnorm = GNORM;
        auto write_output = [&](int otb, int ovalid, int ohv) {
            bf16* ot = sm.OST + (32 * half) * 128 + row;
            if constexpr (gnorm) {
                float ov[32];
                tc::ld32(T_O + lb + 32 * half, ov);
#pragma unroll
                for (int c2 = 0; c2 < 32; ++c2) {
                    const bf16 ob = __float2bfloat16_rn(ov[c2]);
                    ot[c2 * 128] = ob;
                    const float of = __bfloat162float(ob);
                    ov[c2] = of * of;
                }
                sm.ored[warp & 3][32 * half + lane] = reduce_scatter32(ov);
            } else {  // 8 tokens at a time (kept rolled: code size)
#pragma unroll 1
                for (int h8 = 0; h8 < 4; ++h8) {
                    float ov[8];
                    tc::ld8(T_O + lb + 32 * half + 8 * h8, ov);
#pragma unroll
                    for (int c2 = 0; c2 < 8; ++c2) ot[(8 * h8 + c2) * 128] = __float2bfloat16_rn(ov[c2]);
                }
            }
            tc::bar_sync(BAR_S, GS);
            for (int e = gt; e < 64 * 16; e += GS) {
                const int t = e >> 4, ch = e & 15;
                if (t < ovalid) {
                    uint4 val = *reinterpret_cast<const uint4*>(sm.OST + t * 128 + 8 * ch);
                    if constexpr (gnorm) {
                        const float ss = sm.ored[0][t] + sm.ored[1][t] + sm.ored[2][t] + sm.ored[3][t];
                        const float r = rsqrtf(ss * (1.f / 128.f) + p.norm_eps);
                        const uint4 zr = __ldg(reinterpret_cast<const uint4*>(static_cast<const bf16*>(p.z) +
                                                                              (int64_t)(otb + t) * p.ldz + ohv * 128 + 8 * ch));
                        const uint4 wr = __ldg(reinterpret_cast<const uint4*>(static_cast<const bf16*>(p.norm_w) + 8 * ch));
                        const __nv_bfloat162* o2 = reinterpret_cast<const __nv_bfloat162*>(&val);
                        const __nv_bfloat162* z2 = reinterpret_cast<const __nv_bfloat162*>(&zr);
                        const __nv_bfloat162* w2 = reinterpret_cast<const __nv_bfloat162*>(&wr);
                        float y[8];
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const float2 of = __bfloat1622float2(o2[i]), zf = __bfloat1622float2(z2[i]),
                                         wf = __bfloat1622float2(w2[i]);
                            y[2 * i] = wf.x * (of.x * r) * __fdividef(zf.x, 1.f + __expf(-zf.x));
                            y[2 * i + 1] = wf.y * (of.y * r) * __fdividef(zf.y, 1.f + __expf(-zf.y));
                        }
                        val = pack8(y);
                    }
                    *reinterpret_cast<uint4*>(o + (int64_t)(otb + t) * p.ldo + (int64_t)ohv * p.hso + 8 * ch) = val;
                }
            }
        };
        tc::st32_zero(T_O + lb + 32 * half);  // the first product accumulates its o half onto zero
        if (stream_len() == 0 && ok) {  // a job without tokens: its final state is its initial state
            load_state(sm.ring[0], 1.f);
            tc::wait_st();
            store_state(sm.ring[0]);
        }
        tc::wait_st();
        tc::fence_before();
        tc::bar_sync(BAR_S, GS);
        bool w_ready = false;  // W of chunk g is already in shared memory
        bool o_pending = false;  // a chunk's output is still in the o columns
        int o_tb = 0, o_valid = 0, o_hv = 0, o_g = 0;
        int g = 0;             // chunk of the stream
        int len = stream_len();  // chunks in the stream when last read (at least 2 ahead, or all)
        while (ok && g < len) {
            // a job: its initial state (a second half waits for the first's final
            // state), its chunks, its final state
            const JobRec& J = sm.ring[sm.ci[g & 7].jr];
            const int nchj = J.span.y, hvj = J.hv;
            const bool write_o = J.write_o != 0;
            {
                bool fl = true;
                if (J.part == 2 && gt == 0) fl = wait_flag(p.sched + kSchedHeader + J.flag, p.handover_ns, &sm.abort);
                if (!(ok = tc::bar_and(BAR_S, GS, fl))) break;
            }
            for (int c = 0; c < nchj && ok; ++c, ++g) {
                const int s = g & 1;
                if (gt == 0) GDN_STAMP(g, 16);
                // the previous chunk's output (its products are done once the output
                // barrier completes), then its columns back to zero: the first
                // product accumulates its o half onto them.  This overlaps the wait
                // for this chunk's operands.
                if (o_pending) {
                    bool wo = true;
                    if (gt == 0) wo = tc::mbar_wait(&sm.mbar_o, o_g & 1, kSpin, &sm.abort);
                    if (!(ok = tc::bar_and(BAR_S, GS, wo))) break;
                    tc::fence_after();
                    write_output(o_tb, o_valid, o_hv);
                    o_pending = false;
                }
                if (g > 0 && sm.ci[g & 7].write_o) tc::st32_zero(T_O + lb + 32 * half);
                // -Q~ and K~ of this chunk, once the producer has published its
                // factors and read its [rows] K^T columns (while the UT inverse
                // runs), unless done during the previous chunk
                if (!w_ready) {
                    bool rd = true;
                    if (gt == 0) {
                        const volatile int* e1 = &sm.ci[g & 7].eg_ready;
                        const volatile int* e2 = &sm.ci[g & 7].aread;
                        for (uint32_t it = 0; it < kSpin && (*e1 != g || *e2 != g); ++it) {
                            __nanosleep(32);  // yield the issue slots while waiting
                            if ((it & 63) == 63 && *reinterpret_cast<volatile int*>(&sm.abort)) break;
                        }
                        rd = *e1 == g && *e2 == g;
                    }
                    if (!(ok = tc::bar_and(BAR_S, GS, rd))) break;
                    qk_prep_fn(sm, g, gt);
                }
                if (gt == 0) GDN_STAMP(g, 17);
                // chunk g's operands: W/U products done, -Q~ / K~ / A / factors written
                bool gok = true;
                if (gt == 0) gok = tc::mbar_wait(&sm.full[s], (g >> 1) & 1, kSpin, &sm.abort);
                if (!(ok = tc::bar_and(BAR_S, GS, gok))) break;
                tc::fence_after();
                if (gt == 0) GDN_STAMP(g, 18);
                len = stream_len();
                const ChunkInfo& I = sm.ci[g & 7];
                const int tb = I.tb, valid = I.valid;
                const uint32_t T_VNs = s ? T_VN1 : T_VN0;
                if (c == 0) load_state(J, I.eglast);
                if (I.vz) tc::st32_zero(T_VNs + lb + 32 * half);  // no U product: v_new = -W S alone
                const bool w_now = !w_ready;  // W not read during the previous chunk
                if (w_now) w_readout(s);
                w_ready = false;
                tc::wait_st();
                tc::fence_async_smem();
                tc::fence_before();
                tc::bar_sync(BAR_S, GS);
                if (gt == 0) {
                    GDN_STAMP(g, 19);
                    if (w_now) tc::mbar_arrive(&sm.wfree);  // the W columns are free for the next W product
                    tc::fence_after();
                    if (WKST && J.wk_base >= 0) {
                        // the M chain of this summary runs apart: this chunk's W rows,
                        // K~ tile and e^{G_last}, exactly as the products read them
                        const int y = (J.wk_base + c) * 64;
                        const bf16* wsrc = sm.QK[s] + (s ? 64 * 64 : 0);
                        tc::tma_store_2d(&maps.wst, 0, y, wsrc);
                        tc::tma_store_2d(&maps.wst, 64, y, wsrc + 128 * 64);
                        tc::tma_store_2d(&maps.kst, 0, y, sm.KT[s]);
                        tc::tma_store_2d(&maps.kst, 64, y, sm.KT[s] + 64 * 64);
                        tc::bulk_commit();
                        p.wk_eg[J.wk_base + c] = I.eglast;
                    }
                    // [v_new^T | o^T] = [U^T | 0] - S^T [W ; -Q~]^T (slot 0; slot 1 the
                    // other row order), S^T bf16 from tensor memory
                    if (I.write_o) {
                        const uint32_t D1 = s ? T_O : T_VN0;
                        const uint64_t dB = dQK0 + (s ? kQKslot : 0);
#pragma unroll
                        for (int kk = 0; kk < 8; ++kk)
                            tc::mma_ta(D1, T_SB + 8 * kk, dB + tc::koff(128, kk), ID_N128_NEG, 1u);
                    } else {  // no output: v_new^T = U^T - S^T W^T alone (the slot's K rows)
                        const uint64_t dB = dQK0 + krows(s);
#pragma unroll
                        for (int kk = 0; kk < 8; ++kk)
                            tc::mma_ta(T_VNs, T_SB + 8 * kk, dB + tc::koff(128, kk), ID_N64_NEG, 1u);
                    }
                    tc::commit(&sm.mbar_s);
                    GDN_STAMP(g, 20);
                }
                if (!(ok = wait_s())) break;
                if (gt == 0) GDN_STAMP(g, 22);
                // the first product was the last reader of the slot's Q/K tile:
                // refill it with the Q/K of chunk g + 2
                if (WKST && gt == 0 && J.wk_base >= 0) tc::bulk_wait_read();  // the stores have read the slot and K~
                if (gt == 0 && g + 2 < len) issue_qk(g + 2, sm.ci[(g + 2) & 7].tb, sm.ci[(g + 2) & 7].hk);
                {  // v_new^T as bf16 pairs in place (this thread's own columns), the
                   // A operand of the updates
                    float vv[32];
                    tc::ld32(T_VNs + lb + 32 * half, vv);
                    uint32_t w[16];
#pragma unroll
                    for (int j = 0; j < 16; ++j) w[j] = tc::pack_bf16x2(vv[2 * j], vv[2 * j + 1]);
                    tc::stw16(T_VNs + lb + 32 * half, w);
                    tc::wait_st();
                }
                tc::fence_before();
                tc::bar_sync(BAR_S, GS);
                if (gt == 0) {
                    GDN_STAMP(g, 23);
                    tc::fence_after();
                    // S^T <- e^{G_last} S^T + v_new^T K~ (the scaled state is in place);
                    // K step kk of v_new: tokens [16 kk, 16 kk + 16) = columns of half kk / 2
                    const uint64_t dKT = dKT0 + (s ? kKTslot : 0);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        tc::mma_ta(T_S, T_VNs + 32 * (kk >> 1) + 8 * (kk & 1), dKT + tc::mnoff(kk), ID_N128_BMN, 1u);
                    tc::commit(&sm.mbar_s);
                    if (write_o) {  // o^T += v_new^T A^T
                        const uint64_t dAs = dA0 + (s ? kAslot : 0);
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
                            tc::mma_ta(T_O, T_VNs + 32 * (kk >> 1) + 8 * (kk & 1), dAs + tc::koff(64, kk), ID_N64, 1u);
                    }
                    tc::commit(&sm.mbar_o);
                    tc::commit(&sm.afree[s]);
                    GDN_STAMP(g, 24);
                }
                // while it runs: -Q~ / K~ and W of chunk g + 1, if its products are
                // done (then its factors are published and its columns read; the
                // K~ copy must precede the W readout, which overwrites the K rows)
                if (g + 1 < len) {
                    bool rdy = true;
                    if (gt == 0) rdy = tc::mbar_test(&sm.full[s ^ 1], ((g + 1) >> 1) & 1);
                    if (tc::bar_and(BAR_S, GS, rdy)) {
                        tc::fence_after();
                        qk_prep_fn(sm, g + 1, gt);
                        tc::bar_sync(BAR_S, GS);
                        w_readout(s ^ 1);
                        w_ready = true;
                    }
                }
                // e^{G_last} of the next chunk of this job (its gate prefix runs on
                // the producer, published in the chunk's info entry)
                bool eok = true;
                if (c + 1 < nchj && gt == 0) {
                    const volatile int* rdy = &sm.ci[(g + 1) & 7].eg_ready;
                    for (uint32_t it = 0; it < kSpin && *rdy != g + 1; ++it) {
                        __nanosleep(32);
                        if ((it & 63) == 63 && *reinterpret_cast<volatile int*>(&sm.abort)) break;
                    }
                    eok = *rdy == g + 1;
                }
                if (gt == 0) GDN_STAMP(g, 25);
                tc::fence_before();
                if (!(ok = wait_s() && tc::bar_and(BAR_S, GS, eok))) break;
                if (gt == 0 && w_ready) tc::mbar_arrive(&sm.wfree);  // every thread has read chunk g + 1's W
                if (gt == 0) GDN_STAMP(g, 26);
                if (c + 1 < nchj) {
                    // the new state: its bf16 copy, and the state scaled by the next
                    // chunk's e^{G_last}, back into tensor memory (16-column pieces)
                    const float egn = *reinterpret_cast<volatile float*>(&sm.ci[(g + 1) & 7].eglast);
#pragma unroll 1  // kept rolled: the kernel's code size costs instruction-fetch stalls
                    for (int q4 = 0; q4 < 4; ++q4) {
                        float sv[16];
                        uint32_t w[8];
                        tc::ld16(T_S + lb + 64 * half + 16 * q4, sv);
#pragma unroll
                        for (int j = 0; j < 8; ++j) w[j] = tc::pack_bf16x2(sv[2 * j], sv[2 * j + 1]);
                        tc::stw8(T_SB + lb + 32 * half + 8 * q4, w);
#pragma unroll
                        for (int c2 = 0; c2 < 16; ++c2) sv[c2] *= egn;
                        tc::st16(T_S + lb + 64 * half + 16 * q4, sv);
                    }
                } else {
                    store_state(J);
                }
                o_pending = write_o;
                o_tb = tb;
                o_valid = valid;
                o_hv = hvj;
                o_g = g;
                tc::wait_st();
                tc::fence_before();
                tc::bar_sync(BAR_S, GS);
                if (gt == 0) GDN_STAMP(g, 27);
            }
            if (!ok) break;
            if (J.part == 1) {  // hand the final state to the second half
                if (gt == 0 && !p.no_publish) {
                    __threadfence();
                    st_release(p.sched + kSchedHeader + J.flag, 1);
                }
            }
            tc::bar_sync(BAR_S, GS);
            if (gt == 0) *reinterpret_cast<volatile int*>(&sm.jdone) += 1;  // the job's ring entry is free
        }
        if (ok && o_pending) {  // the last chunk's output
            bool wo = true;
            if (gt == 0) wo = tc::mbar_wait(&sm.mbar_o, o_g & 1, kSpin, &sm.abort);
            if ((ok = tc::bar_and(BAR_S, GS, wo))) {
                tc::fence_after();
                write_output(o_tb, o_valid, o_hv);
            }
        }
        if (!ok && gt == 0) *reinterpret_cast<volatile int*>(&sm.abort) = 1;
        if (tid == GS) {  // every product and store this thread issued has completed
            tc::commit(&sm.fin_s);
            tc::mbar_wait(&sm.fin_s, 0, kSpin);
            if (WKST) tc::bulk_wait();
        }
    }
    if (!ok && gt == 0) {
        atomicAdd(&g_gdn_timeouts, 1);
        if (p.status) atomicCAS(p.status, 0, (int)GDN_ERR_TIMEOUT);
    }
    tc::fence_before();
    __syncthreads();
    if (tid == 0) {  // copies still in flight after an early exit land before the memory is released
        for (int ss = 0; ss < 2; ++ss)
            if (sm.qk_issued[ss] > sm.qk_waited[ss]) tc::mbar_wait(&sm.ld_qk[ss], (sm.qk_issued[ss] - 1) & 1, kSpin);
        if (sm.v_issued > sm.v_waited) tc::mbar_wait(&sm.ld_v, (sm.v_issued - 1) & 1, kSpin);
    }
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc(tmem, 512);
    empty_sequences_final(p, src);
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
static gdn_status make_map(CUtensorMap* m, const void* base, int64_t ld, int64_t cols, int64_t rows);
gdn_status make_map_bf16(CUtensorMap* m, const void* base, int64_t ld, int64_t cols, int64_t rows) {
    return make_map(m, base, ld, cols, rows);
}
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

// Split-item hand-over settings (a testing hook, gdn_debug_set_handover).
static long long g_handover_ns = 1000000000ll;
static int g_handover_publish = 1;
static int g_split_items = 1;  // work-queue splitting of items (gdn_debug_set_split)

gdn_status launch_chunk_tc(ChunkParams p, int src, dim3 grid, cudaStream_t s) {
    p.handover_ns = g_handover_ns;
    p.no_publish = g_handover_publish ? 0 : 1;
    const size_t smem = sizeof(SmemWS) + 1024;
    // three instantiations: the gated-norm epilogue (the layer), the stores of a
    // summary's W rows / K~ for the M chains run apart (shard pass 1), and plain
    const bool wkst = !p.z && p.m_external && p.wk_w && src == JOBS_SHARD_PASS1;
    const void* fn = p.z ? (const void*)chunk_tc_kernel<true, false>
                         : (wkst ? (const void*)chunk_tc_kernel<false, true> : (const void*)chunk_tc_kernel<false, false>);
    gdn_status st = set_smem_attr(fn, smem);
    if (st != GDN_OK) return st;
    TmaMaps maps;
    memset(&maps, 0, sizeof(maps));
    if (p.T > 0 && !p.head_major) {
        if ((st = make_map(&maps.q, p.q, p.ldq, (int64_t)p.Hk * 128, p.T)) != GDN_OK) return st;
        if ((st = make_map(&maps.k, p.k, p.ldk, (int64_t)p.Hk * 128, p.T)) != GDN_OK) return st;
        if ((st = make_map(&maps.v, p.v, p.ldv, (int64_t)p.Hv * 128, p.T)) != GDN_OK) return st;
    } else if (p.T > 0) {  // dense head-major [H, T, 128]: [H*T rows x 128 columns]
        if ((st = make_map(&maps.q, p.q, 128, 128, (int64_t)p.Hk * p.T)) != GDN_OK) return st;
        if ((st = make_map(&maps.k, p.k, 128, 128, (int64_t)p.Hk * p.T)) != GDN_OK) return st;
        if ((st = make_map(&maps.v, p.v, 128, 128, (int64_t)p.Hv * p.T)) != GDN_OK) return st;
    }
    if (p.m_external && p.wk_w && p.wk_kt) {  // stored W rows / K~: [P * Hv * wk_nch * 64 rows x 128]
        const int64_t rows = (int64_t)p.n_shards * p.Hv * p.wk_nch * 64;
        if ((st = make_map(&maps.wst, p.wk_w, 128, 128, rows)) != GDN_OK) return st;
        if ((st = make_map(&maps.kst, p.wk_kt, 128, 128, rows)) != GDN_OK) return st;
    }
    if (p.sched && grid.x > (unsigned)kMaxLptItems) p.sched = nullptr;  // beyond the order kernel's scratch
    if (!p.status && p.sched) p.status = p.sched + 2;  // the work queue's status word
    if (p.sched) {  // work queue: the order of the entries, then one persistent CTA per SM
        static int sms[64];
        int dev = 0;
        if (cudaGetDevice(&dev) == cudaSuccess && dev >= 0 && dev < 64) {
            if (!sms[dev]) cudaDeviceGetAttribute(&sms[dev], cudaDevAttrMultiProcessorCount, dev);
            p.num_sms = sms[dev];
        }
        p.sched_items = (int)grid.x;
        p.sched_m = (int)(grid.y * grid.z);
        p.sched_ny = (int)grid.y;
        // halves for single-segment launches with final states; short tails for
        // the shard passes (every split part has a hand-over destination there,
        // else its first part runs whole)
        int rule = kSplitNone;
        if (!g_split_items) rule = kSplitNone;
        else if (p.h_final != nullptr && (src == JOBS_SEQS || (src == JOBS_SHARD_PASS1 && p.n_shards == 1)))
            rule = kSplitHalves;
        else if (p.n_shards > 1 && (src == JOBS_SHARD_PASS1 || src == JOBS_SHARD_PASS2))
            rule = kSplitTail;
        if ((st = launch_chunk_order(p, src, p.sched_items, p.sched_m, rule, s)) != GDN_OK) return st;
        const long long jobs = 2ll * p.sched_items * p.sched_m;
        grid = dim3((unsigned)(jobs < p.num_sms ? jobs : (p.num_sms > 0 ? p.num_sms : 1)), 1, 1);
    }
    if (p.z) chunk_tc_kernel<true, false><<<grid, NT, smem, s>>>(p, src, maps);
    else if (wkst) chunk_tc_kernel<false, true><<<grid, NT, smem, s>>>(p, src, maps);
    else chunk_tc_kernel<false, false><<<grid, NT, smem, s>>>(p, src, maps);
    return check_launch("chunk_tc_kernel");
}

}  // namespace gdn

extern "C" gdn_status gdn_debug_set_split(int32_t enable) {
    gdn::g_split_items = enable ? 1 : 0;
    return GDN_OK;
}

extern "C" gdn_status gdn_debug_set_handover(int64_t wait_ns, int publish) {
    if (wait_ns < 0) return gdn::fail(GDN_ERR_INVALID_ARG, "wait_ns=%lld < 0", (long long)wait_ns);
    gdn::g_handover_ns = wait_ns;
    gdn::g_handover_publish = publish ? 1 : 0;
    return GDN_OK;
}

#ifdef GDN_PHASE_STAMPS
extern "C" int gdn_debug_phase_stamps(long long* out, int n) {
    if (n > gdn::kStampN * 32) n = gdn::kStampN * 32;
    if (cudaMemcpyFromSymbol(out, gdn::g_gdn_stamps, sizeof(long long) * n) != cudaSuccess) return -1;
    return n;
}
#endif
