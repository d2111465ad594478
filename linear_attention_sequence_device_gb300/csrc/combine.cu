// Cross-shard prefix merge of the affine state summaries (hyper-parallel
// page, _merge_gdn_prefix_state_summaries_torch; _apply_gdn_state_summary):
//   S_in[0] = S0 or 0;  S_in[r] = M[r-1] S_in[r-1] + N[r-1]
// Sequential over shards in fp32, as the page's loop; parallel over value
// heads and 16- or 32-column tiles of the state (16 while the CTAs still fit
// the SMs: the sequential steps then run on twice as many SMs).  In the sharded forward each
// shard's carry is classified from the plan: affine (M, N) for a shard that
// a single sequence spans from an earlier shard into a later one, constant
// (N only, M = 0) when the carried sequence starts inside the shard, and
// none when the next shard starts a new sequence.
#include "chunk_common.cuh"
#include "gdn_internal.cuh"

namespace gdn {
gdn_status set_smem_attr(const void* func, size_t bytes);
namespace {

constexpr int NT = 256;

// grid (Hv, dv / CT), 256 threads.  Thread = state column c0 + tid % CT and
// row group tid / CT (CG = 256 / CT groups of DK / CG rows).  Each shard's M
// (DK x DK fp32) is staged in shared memory with cp.async, the next one in
// flight while the current is applied (the loads are the only global traffic
// on the sequential path); reads of M are broadcasts (one row element for the
// threads of a row group), reads of S are one column per thread.
template <int DK, int CT>
__global__ void __launch_bounds__(NT) combine_kernel(const float* __restrict__ M,
                                                     const float* __restrict__ N,
                                                     const float* __restrict__ S0, int P, int Hv,
                                                     int dv, float* __restrict__ S_in,
                                                     const int32_t* __restrict__ plan) {
    extern __shared__ __align__(16) float csm[];
    float* Ms = csm;                // [2][DK * DK]
    float* S = csm + 2 * DK * DK;   // [DK][CT]
    if (plan && plan[0] != 0) return;
    constexpr int CG = NT / CT;     // row groups
    constexpr int RPW = DK / CG;    // rows per group
    const int h = blockIdx.x, c0 = blockIdx.y * CT;
    const int tid = threadIdx.x, lane = tid % CT, warp = tid / CT;
    const int64_t hs = (int64_t)DK * dv;
    // 2 = affine (M, N), 1 = constant (N only, M = 0), 0 = none
    auto kind = [&](int r) -> int {
        if (!plan) return 2;
        const int32_t* rec = plan + GDN_PLAN_REC(r);
        if (rec[GDN_PLAN_POST_NUM_RANKS] == 0) return 0;
        return (rec[GDN_PLAN_LOCAL_NUM_SEQS] == 1 && !rec[GDN_PLAN_IS_FIRST_RANK]) ? 2 : 1;
    };
    auto stage = [&](int r) {  // M of shard r into buffer r & 1 (one cp.async group, maybe empty)
        if (r < P - 1 && kind(r) == 2) {
            const float* src = M + ((int64_t)r * Hv + h) * DK * DK;
            float* dst = Ms + (r & 1) * DK * DK;
            for (int e = tid; e < DK * DK / 4; e += NT) cp_async16(dst + 4 * e, src + 4 * e, 16);
        }
        cp_async_commit();
    };
    for (int i = warp; i < DK; i += CG) S[i * CT + lane] = S0 ? S0[h * hs + (int64_t)i * dv + c0 + lane] : 0.f;
    stage(0);
    __syncthreads();
    for (int r = 0; r < P; ++r) {
        float* out = S_in + ((int64_t)r * Hv + h) * hs;
        for (int i = warp; i < DK; i += CG) out[(int64_t)i * dv + c0 + lane] = S[i * CT + lane];
        if (r == P - 1) break;
        const int kd = kind(r);
        stage(r + 1);  // the next shard's M streams in while this one is applied
        float acc[RPW];
        const float* Nr = N + ((int64_t)r * Hv + h) * hs + c0 + lane;
#pragma unroll
        for (int j = 0; j < RPW; ++j) acc[j] = kd >= 1 ? Nr[(int64_t)(warp * RPW + j) * dv] : 0.f;
        if (kd == 2) {
            cp_async_wait<1>();  // this shard's M has landed
            __syncthreads();
            const float* Mr = Ms + (r & 1) * DK * DK + warp * RPW * DK;
#pragma unroll 2
            for (int m = 0; m < DK; m += 4) {
                const float s0 = S[(m + 0) * CT + lane], s1 = S[(m + 1) * CT + lane];
                const float s2 = S[(m + 2) * CT + lane], s3 = S[(m + 3) * CT + lane];
#pragma unroll
                for (int j = 0; j < RPW; ++j) {
                    const float4 mv = *reinterpret_cast<const float4*>(Mr + j * DK + m);
                    acc[j] = fmaf(mv.x, s0, fmaf(mv.y, s1, fmaf(mv.z, s2, fmaf(mv.w, s3, acc[j]))));
                }
            }
        }
        __syncthreads();  // every warp is done reading S and this M
#pragma unroll
        for (int j = 0; j < RPW; ++j) S[(warp * RPW + j) * CT + lane] = acc[j];
        __syncthreads();
    }
    cp_async_wait_all();
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

template <int CT>
static gdn_status launch_combine_ct(const float* M, const float* N, const float* S0, int P, int Hv, int dk, int dv,
                                   float* S_in, const int32_t* plan, cudaStream_t s) {
    dim3 grid(Hv, dv / CT);
    const size_t smem = sizeof(float) * (2 * (size_t)dk * dk + (size_t)dk * CT);
    gdn_status st;
    switch (dk) {
        case 32:
            combine_kernel<32, CT><<<grid, NT, smem, s>>>(M, N, S0, P, Hv, dv, S_in, plan);
            break;
        case 64:
            if ((st = set_smem_attr((const void*)combine_kernel<64, CT>, smem)) != GDN_OK) return st;
            combine_kernel<64, CT><<<grid, NT, smem, s>>>(M, N, S0, P, Hv, dv, S_in, plan);
            break;
        case 128:
            if ((st = set_smem_attr((const void*)combine_kernel<128, CT>, smem)) != GDN_OK) return st;
            combine_kernel<128, CT><<<grid, NT, smem, s>>>(M, N, S0, P, Hv, dv, S_in, plan);
            break;
        default: return fail(GDN_ERR_UNSUPPORTED_SHAPE, "dk=%d", dk);
    }
    return check_launch("combine_kernel");
}

gdn_status launch_combine(const float* M, const float* N, const float* S0, int P, int Hv, int dk,
                          int dv, float* S_in, const int32_t* plan, cudaStream_t s) {
    if ((int64_t)Hv * (dv / 16) <= device_sm_count())
        return launch_combine_ct<16>(M, N, S0, P, Hv, dk, dv, S_in, plan, s);
    return launch_combine_ct<32>(M, N, S0, P, Hv, dk, dv, S_in, plan, s);
}

gdn_status launch_empty_seq_final(const int32_t* cu, int num_seqs, int Hv, int dk, int dv,
                                  const float* h0, float* h_final, const int32_t* plan,
                                  cudaStream_t s) {
    empty_seq_final_kernel<<<num_seqs, 256, 0, s>>>(cu, Hv, dk, dv, h0, h_final, plan);
    return check_launch("empty_seq_final_kernel");
}

}  // namespace gdn
