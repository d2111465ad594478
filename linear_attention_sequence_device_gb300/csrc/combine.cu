// Cross-shard prefix merge of the affine state summaries (hyper-parallel
// page, _merge_gdn_prefix_state_summaries_torch; _apply_gdn_state_summary):
//   S_in[0] = S0 or 0;  S_in[r] = M[r-1] S_in[r-1] + N[r-1]
// Sequential over shards in fp32, as the page's loop; parallel over value
// heads and 32-column tiles of the state.  In the sharded forward each
// shard's carry is classified from the plan: affine (M, N) for a shard that
// a single sequence spans from an earlier shard into a later one, constant
// (N only, M = 0) when the carried sequence starts inside the shard, and
// none when the next shard starts a new sequence.
#include "gdn_internal.cuh"

namespace gdn {
namespace {

constexpr int NT = 256;
constexpr int CT = 32;

template <int DK>
__global__ void __launch_bounds__(NT) combine_kernel(const float* __restrict__ M,
                                                     const float* __restrict__ N,
                                                     const float* __restrict__ S0, int P, int Hv,
                                                     int dv, float* __restrict__ S_in,
                                                     const int32_t* __restrict__ plan) {
    constexpr int dk = DK;
    __shared__ float S[DK][CT + 1];
    if (plan && plan[0] != 0) return;
    const int h = blockIdx.x, c0 = blockIdx.y * CT;
    const int tid = threadIdx.x;
    constexpr int tpr = NT / DK;      // threads per state row
    constexpr int cpt = CT / tpr;     // columns per thread
    const int row = tid / tpr, cs = (tid % tpr) * cpt;
    const int64_t hs = (int64_t)dk * dv;
    for (int e = tid; e < dk * CT; e += NT) {
        const int i = e / CT, c = e % CT;
        S[i][c] = S0 ? S0[h * hs + (int64_t)i * dv + c0 + c] : 0.f;
    }
    __syncthreads();
    for (int r = 0; r < P; ++r) {
        float* out = S_in + ((int64_t)r * Hv + h) * hs;
        for (int e = tid; e < dk * CT; e += NT) {
            const int i = e / CT, c = e % CT;
            out[(int64_t)i * dv + c0 + c] = S[i][c];
        }
        if (r == P - 1) break;
        int kind = 2;  // 2 = affine, 1 = constant, 0 = none
        if (plan) {
            const int32_t* rec = plan + GDN_PLAN_REC(r);
            if (rec[GDN_PLAN_POST_NUM_RANKS] == 0) kind = 0;
            else if (rec[GDN_PLAN_LOCAL_NUM_SEQS] == 1 && !rec[GDN_PLAN_IS_FIRST_RANK]) kind = 2;
            else kind = 1;
        }
        float acc[cpt];
        const float* Nr = N + ((int64_t)r * Hv + h) * hs + (int64_t)row * dv + c0 + cs;
#pragma unroll
        for (int c = 0; c < cpt; ++c) acc[c] = (kind >= 1) ? Nr[c] : 0.f;
        if (kind == 2) {
            const float* Mr = M + ((int64_t)r * Hv + h) * dk * dk + (int64_t)row * dk;
            for (int m = 0; m < dk; ++m) {
                const float a = __ldg(Mr + m);
#pragma unroll
                for (int c = 0; c < cpt; ++c) acc[c] = fmaf(a, S[m][cs + c], acc[c]);
            }
        }
        __syncthreads();
#pragma unroll
        for (int c = 0; c < cpt; ++c) S[row][cs + c] = acc[c];
        __syncthreads();
    }
}

__global__ void empty_seq_final_kernel(const int32_t* __restrict__ cu, int Hv, int dk, int dv,
                                       const float* __restrict__ h0, float* __restrict__ h_final,
                                       const int32_t* __restrict__ plan) {
    if (plan && plan[0] != 0) return;
    const int n = blockIdx.x;
    if (cu[n] != cu[n + 1]) return;
    const int64_t sz = (int64_t)Hv * dk * dv;
    for (int64_t e = threadIdx.x; e < sz; e += blockDim.x)
        h_final[n * sz + e] = h0 ? h0[n * sz + e] : 0.f;
}

// Gated RMS norm in place, one warp per (token, value head) row of dv
// values (the wrappers' norm(core_attn_out, z) on rows of head_v_dim):
// o <- w * o / sqrt(mean(o^2) + eps) * silu(z); the tensor-core chunk kernel
// applies the same as its output epilogue instead.
template <typename E>
__global__ void gated_norm_kernel(E* __restrict__ o, const E* __restrict__ z, int64_t ldz, const E* __restrict__ w,
                                  float eps, int64_t rows, int Hv, int dv) {
    const int lane = threadIdx.x & 31;
    const int64_t r = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (r >= rows) return;
    const int64_t t = r / Hv;
    const int h = (int)(r - t * Hv);
    E* orow = o + r * dv;
    const E* zrow = z + t * ldz + (int64_t)h * dv;
    float ss = 0.f;
    for (int d = lane; d < dv; d += 32) {
        const float x = Elem<E>::to_f(orow[d]);
        ss = fmaf(x, x, ss);
    }
#pragma unroll
    for (int off = 16; off; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
    const float inv = rsqrtf(ss / (float)dv + eps);
    for (int d = lane; d < dv; d += 32) {
        const float zz = Elem<E>::to_f(zrow[d]);
        const float y = Elem<E>::to_f(w[d]) * (Elem<E>::to_f(orow[d]) * inv) * (zz / (1.f + expf(-zz)));
        orow[d] = Elem<E>::from_f(y);
    }
}

}  // namespace

gdn_status launch_gated_norm(void* o, const void* z, int64_t ldz, const void* w, float eps, int64_t T, int Hv,
                             int dv, gdn_dtype dt, cudaStream_t s) {
    const int64_t rows = T * Hv;
    if (rows == 0) return GDN_OK;
    const int wpb = 8;
    const unsigned blocks = (unsigned)((rows + wpb - 1) / wpb);
    if (dt == GDN_BF16)
        gated_norm_kernel<__nv_bfloat16><<<blocks, 32 * wpb, 0, s>>>(
            static_cast<__nv_bfloat16*>(o), static_cast<const __nv_bfloat16*>(z), ldz,
            static_cast<const __nv_bfloat16*>(w), eps, rows, Hv, dv);
    else
        gated_norm_kernel<float><<<blocks, 32 * wpb, 0, s>>>(static_cast<float*>(o), static_cast<const float*>(z),
                                                             ldz, static_cast<const float*>(w), eps, rows, Hv, dv);
    return check_launch("gated_norm_kernel");
}

gdn_status launch_combine(const float* M, const float* N, const float* S0, int P, int Hv, int dk,
                          int dv, float* S_in, const int32_t* plan, cudaStream_t s) {
    dim3 grid(Hv, dv / CT);
    switch (dk) {
        case 32: combine_kernel<32><<<grid, NT, 0, s>>>(M, N, S0, P, Hv, dv, S_in, plan); break;
        case 64: combine_kernel<64><<<grid, NT, 0, s>>>(M, N, S0, P, Hv, dv, S_in, plan); break;
        case 128: combine_kernel<128><<<grid, NT, 0, s>>>(M, N, S0, P, Hv, dv, S_in, plan); break;
        default: return fail(GDN_ERR_UNSUPPORTED_SHAPE, "dk=%d", dk);
    }
    return check_launch("combine_kernel");
}

gdn_status launch_empty_seq_final(const int32_t* cu, int num_seqs, int Hv, int dk, int dv,
                                  const float* h0, float* h_final, const int32_t* plan,
                                  cudaStream_t s) {
    empty_seq_final_kernel<<<num_seqs, 256, 0, s>>>(cu, Hv, dk, dv, h0, h_final, plan);
    return check_launch("empty_seq_final_kernel");
}

}  // namespace gdn
