// Device pieces shared by the bf16 (tensor-core) and fp32 (FFMA) chunk kernels.
//
// The chunked WY/UT form of the gated delta rule (hyper-parallel page,
// _prepare_gdn_chunks_for_summary): inside a chunk of C = 64 tokens with
// in-chunk gate prefix G_i = sum_{j<=i} g_j,
//   L = strict_lower(diag(beta) (K K^T) o Gamma),  Gamma_ij = exp(G_i - G_j)
//   T = (I + L)^-1            (the page forms it by forward substitution)
//   W = T diag(beta exp(G)) K,   U = T diag(beta) V
// and across chunks (_run_prepared_gdn_chunks):
//   v_new = U - W S
//   o     = scale (exp(G) o Q) S + (scale Q K^T o Gamma_incl) v_new
//   S    <- exp(G_last) S + (K o exp(G_last - G))^T v_new
#pragma once

#include "gdn_internal.cuh"

namespace gdn {

// ---- cp.async helpers -------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
// 16-byte async copy global -> shared; src_bytes == 0 writes zeros.
__device__ __forceinline__ void cp_async16(void* dst, const void* src, int src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(smem_u32(dst)),
                 "l"(src), "r"(src_bytes));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;\n" ::); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N)); }

// ---- gate prefix -------------------------------------------------------------
// Warp 0: G = inclusive cumsum of g over the chunk (2 values per lane), then
//   Gs[i] = G_i, eG[i] = exp(G_i), eGl[i] = exp(G_63 - G_i).
// Rows past the segment end carry g = 0, so G_63 is the last valid row's G.
__device__ __forceinline__ void gate_prefix_warp0(const float* g_in, float* Gs, float* eG,
                                                  float* eGl) {
    const int lane = threadIdx.x & 31;
    float a = g_in[2 * lane], b = g_in[2 * lane + 1];
    float s = a + b;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        float t = __shfl_up_sync(0xffffffffu, s, off);
        if (lane >= off) s += t;
    }
    const float G1 = s;        // inclusive through element 2*lane+1
    const float G0 = s - b;    // inclusive through element 2*lane
    const float Gl = __shfl_sync(0xffffffffu, s, 31);
    Gs[2 * lane] = G0;
    Gs[2 * lane + 1] = G1;
    eG[2 * lane] = expf(G0);
    eG[2 * lane + 1] = expf(G1);
    eGl[2 * lane] = expf(Gl - G0);
    eGl[2 * lane + 1] = expf(Gl - G1);
}

// ---- unit lower-triangular inverse --------------------------------------------
// Ts = (I + Ls)^-1 for a strictly lower 64x64 Ls (row stride LD floats), in
// fp32, by 16x16 blocks: each diagonal block by forward substitution, then the
// off-diagonal blocks level by level,
//   T_ab = -T_aa sum_{m=b}^{a-1} L_am T_mb      (a > b).
// Xs: scratch of 3*16*17 floats.  All NT threads must call this.
template <int NT, int LD>
__device__ __forceinline__ void unit_lower_inverse64(const float* Ls, float* Ts, float* Xs) {
    const int tid = threadIdx.x;
    // zero the strictly-upper blocks of Ts
    for (int e = tid; e < 64 * 64; e += NT) {
        int i = e >> 6, j = e & 63;
        if ((i >> 4) < (j >> 4)) Ts[i * LD + j] = 0.f;
    }
    if (tid < 64) {
        const int b = tid >> 4, c = tid & 15;
        const float* L = Ls + (16 * b) * LD + 16 * b;
        float x[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            float acc = (i == c) ? 1.f : 0.f;
#pragma unroll
            for (int m = 0; m < i; ++m) acc = fmaf(-L[i * LD + m], (m >= c) ? x[m] : 0.f, acc);
            x[i] = (i >= c) ? acc : 0.f;
        }
        float* Td = Ts + (16 * b) * LD + 16 * b;
#pragma unroll
        for (int i = 0; i < 16; ++i) Td[i * LD + c] = x[i];
    }
    __syncthreads();
#pragma unroll 1
    for (int d = 1; d < 4; ++d) {
        const int nblk = 4 - d;
        for (int e = tid; e < nblk * 256; e += NT) {
            const int b = e >> 8, i = (e >> 4) & 15, j = e & 15;
            const int a = b + d;
            const float* Lrow = Ls + (16 * a + i) * LD;
            float acc = 0.f;
            for (int m = 16 * b; m < 16 * a; ++m) acc = fmaf(Lrow[m], Ts[m * LD + 16 * b + j], acc);
            Xs[(b * 16 + i) * 17 + j] = acc;
        }
        __syncthreads();
        for (int e = tid; e < nblk * 256; e += NT) {
            const int b = e >> 8, i = (e >> 4) & 15, j = e & 15;
            const int a = b + d;
            const float* Drow = Ts + (16 * a + i) * LD + 16 * a;
            float acc = 0.f;
            for (int m = 0; m <= i; ++m) acc = fmaf(Drow[m], Xs[(b * 16 + m) * 17 + j], acc);
            Ts[(16 * a + i) * LD + 16 * b + j] = -acc;
        }
        __syncthreads();
    }
}

}  // namespace gdn

namespace gdn {

// ---- tf32 tensor-core block products (m16n8k8 mma.sync) -------------------
__device__ __forceinline__ uint32_t to_tf32(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return r;
}
__device__ __forceinline__ void mma_tf32(float* d, const uint32_t* a, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

}  // namespace gdn

namespace gdn {

// acc (16x16, two m16n8 accumulators) += A (16x16 block at Ab) * B (16x16 block
// at Bb), both fp32 in shared memory with row stride LD, as tf32 products.
template <int LD>
__device__ __forceinline__ void mma_block16_tf32(float (&acc)[2][4], const float* Ab, const float* Bb) {
    const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
#pragma unroll
    for (int kk = 0; kk < 16; kk += 8) {
        const float* Ar = Ab + g * LD + kk + t;
        uint32_t af[4] = {to_tf32(Ar[0]), to_tf32(Ar[8 * LD]), to_tf32(Ar[4]), to_tf32(Ar[8 * LD + 4])};
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            const float* Br = Bb + (kk + t) * LD + 8 * nt + g;
            mma_tf32(acc[nt], af, to_tf32(Br[0]), to_tf32(Br[4 * LD]));
        }
    }
}
// Write -acc (16x16) to the block at Cb.
template <int LD>
__device__ __forceinline__ void store_block16_neg(const float (&acc)[2][4], float* Cb) {
    const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
        float* Cr = Cb + g * LD + 8 * nt + 2 * t;
        *reinterpret_cast<float2*>(Cr) = make_float2(-acc[nt][0], -acc[nt][1]);
        *reinterpret_cast<float2*>(Cr + 8 * LD) = make_float2(-acc[nt][2], -acc[nt][3]);
    }
}
template <int LD>
__device__ __forceinline__ void store_block16(const float (&acc)[2][4], float* Cb) {
    const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
        float* Cr = Cb + g * LD + 8 * nt + 2 * t;
        *reinterpret_cast<float2*>(Cr) = make_float2(acc[nt][0], acc[nt][1]);
        *reinterpret_cast<float2*>(Cr + 8 * LD) = make_float2(acc[nt][2], acc[nt][3]);
    }
}

}  // namespace gdn
