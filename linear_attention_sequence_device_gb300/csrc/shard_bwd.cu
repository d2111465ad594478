// The backward across virtual shards (hyper-parallel page
// linear_attention_context_parallel.py: _RecvInitialStateP2PFunction /
// _SendFinalStateP2PFunction, whose backward sends the state gradient from a
// shard to the one before it).
//
// The sequences are cut at the shard boundaries into segments (the shard
// plan's local segments).  A segment's state map is affine,
// S_end = M S_start + N, so its backward is linear in its end-state gradient:
// dS_start = M^T dS_end + b, where b is the start-state gradient it gets from
// its own outputs alone (dS_end = 0).  With every segment's S_start known
// (forward merge of the summaries), one backward pass over the segments with
// dS_end = 0 gives b; a reverse merge over each sequence's segments,
//   dS_end(last) = dh_final,  dS_end(j - 1) = dS_start(j) = M_j^T dS_end(j) + b_j,
// gives every segment's true end-state gradient; a second backward pass with
// it gives the input gradients.  This file holds the segment list and the two
// merges; the passes are the backward kernel's.
#include "gdn_internal.cuh"

namespace gdn {
namespace {

constexpr int kMergeThreads = 256;
constexpr int kTile = 32;  // state columns per merge block

// the plan's local segments of all shards, in token order: cu_seg [nmax + 1]
// (padded with T: empty segments), seg_seq [nmax] (global sequence, -1 for padding)
__global__ void segments_kernel(const int32_t* __restrict__ plan, int num_seqs, int P, int T, int nmax,
                                int32_t* __restrict__ cu_seg, int32_t* __restrict__ seg_seq) {
    if (plan[0] != 0) {  // malformed cu_seqlens (the status word says so): no segment has tokens
        if (blockIdx.x == 0)
            for (int j = threadIdx.x; j <= nmax; j += blockDim.x) {
                cu_seg[j] = 0;
                if (j < nmax) seg_seq[j] = -1;
            }
        return;
    }
    const int part = T / P;
    for (int r = blockIdx.x; r < P; r += gridDim.x) {
        const int32_t* rec = plan + GDN_PLAN_REC(r);
        const int cnt = rec[GDN_PLAN_LOCAL_NUM_SEQS], off = rec[GDN_PLAN_SEG_OFFSET];
        const int32_t* lc = plan + GDN_PLAN_CU(num_seqs, P, r);
        const int32_t* ls = plan + GDN_PLAN_SEQ(num_seqs, P, r);
        for (int j = threadIdx.x; j < cnt; j += blockDim.x) {
            cu_seg[off + j] = r * part + lc[j];
            seg_seq[off + j] = ls[j];
        }
        if (r == P - 1 && threadIdx.x == 0) {
            for (int j = off + cnt; j <= nmax; ++j) cu_seg[j] = T;
            for (int j = off + cnt; j < nmax; ++j) seg_seq[j] = -1;
        }
    }
}

// Per (sequence, value head, 32-column tile): the first and one-past-last
// segment of the sequence (segments of a sequence are consecutive).
__device__ void seq_segments(const int32_t* seg_seq, int nmax, int n, int& j0, int& j1) {
    __shared__ int lo, hi;
    if (threadIdx.x == 0) { lo = nmax; hi = -1; }
    __syncthreads();
    for (int j = threadIdx.x; j < nmax; j += blockDim.x)
        if (seg_seq[j] == n) { atomicMin(&lo, j); atomicMax(&hi, j); }
    __syncthreads();
    j0 = lo;
    j1 = hi + 1;
    __syncthreads();
}

// forward merge: S_start(first) = h0 (or 0), S_start(j + 1) = M_j S_start(j) + N_j
template <int DK, int DV>
__global__ void __launch_bounds__(kMergeThreads) seg_merge_fwd_kernel(
    const int32_t* __restrict__ plan, const int32_t* __restrict__ seg_seq, int nmax, int Hv,
    const float* __restrict__ M, const float* __restrict__ N, const float* __restrict__ h0,
    float* __restrict__ S_start) {
    if (plan[0] != 0) return;
    __shared__ float S[DK][kTile];
    const int n = blockIdx.x, hv = blockIdx.y, c0 = blockIdx.z * kTile;
    int j0, j1;
    seq_segments(seg_seq, nmax, n, j0, j1);
    for (int e = threadIdx.x; e < DK * kTile; e += kMergeThreads) {
        const int i = e / kTile, c = e % kTile;
        S[i][c] = h0 ? h0[(((int64_t)n * Hv + hv) * DK + i) * DV + c0 + c] : 0.f;
    }
    __syncthreads();
    for (int j = j0; j < j1; ++j) {
        const int64_t base = (int64_t)j * Hv + hv;
        const float* Mj = M + base * DK * DK;
        const float* Nj = N + base * DK * DV;
        float acc[DK * kTile / kMergeThreads];
#pragma unroll
        for (int q = 0; q < DK * kTile / kMergeThreads; ++q) {
            const int e = threadIdx.x + q * kMergeThreads, i = e / kTile, c = e % kTile;
            S_start[(base * DK + i) * DV + c0 + c] = S[i][c];
            float s = Nj[(int64_t)i * DV + c0 + c];
            for (int k = 0; k < DK; ++k) s = fmaf(__ldg(Mj + (int64_t)i * DK + k), S[k][c], s);
            acc[q] = s;
        }
        __syncthreads();
#pragma unroll
        for (int q = 0; q < DK * kTile / kMergeThreads; ++q) {
            const int e = threadIdx.x + q * kMergeThreads;
            S[e / kTile][e % kTile] = acc[q];
        }
        __syncthreads();
    }
}

// reverse merge: dS_end(last) = dh_final (or 0), dS_end(j - 1) = M_j^T dS_end(j) + b_j
template <int DK, int DV>
__global__ void __launch_bounds__(kMergeThreads) seg_merge_bwd_kernel(
    const int32_t* __restrict__ plan, const int32_t* __restrict__ seg_seq, int nmax, int Hv,
    const float* __restrict__ M, const float* __restrict__ b, const float* __restrict__ dh_final,
    float* __restrict__ dS_end) {
    if (plan[0] != 0) return;
    __shared__ float D[DK][kTile];
    const int n = blockIdx.x, hv = blockIdx.y, c0 = blockIdx.z * kTile;
    int j0, j1;
    seq_segments(seg_seq, nmax, n, j0, j1);
    for (int e = threadIdx.x; e < DK * kTile; e += kMergeThreads) {
        const int i = e / kTile, c = e % kTile;
        D[i][c] = dh_final ? dh_final[(((int64_t)n * Hv + hv) * DK + i) * DV + c0 + c] : 0.f;
    }
    __syncthreads();
    for (int j = j1 - 1; j >= j0; --j) {
        const int64_t base = (int64_t)j * Hv + hv;
        const float* Mj = M + base * DK * DK;
        const float* bj = b + base * DK * DV;
        float acc[DK * kTile / kMergeThreads];
#pragma unroll
        for (int q = 0; q < DK * kTile / kMergeThreads; ++q) {
            const int e = threadIdx.x + q * kMergeThreads, k = e / kTile, c = e % kTile;
            dS_end[(base * DK + k) * DV + c0 + c] = D[k][c];
            float s = bj[(int64_t)k * DV + c0 + c];
            for (int i = 0; i < DK; ++i) s = fmaf(__ldg(Mj + (int64_t)i * DK + k), D[i][c], s);
            acc[q] = s;
        }
        __syncthreads();
#pragma unroll
        for (int q = 0; q < DK * kTile / kMergeThreads; ++q) {
            const int e = threadIdx.x + q * kMergeThreads;
            D[e / kTile][e % kTile] = acc[q];
        }
        __syncthreads();
    }
}

// dh0 of each sequence: the start-state gradient of its first segment, or,
// for a sequence without tokens, dh_final (or 0)
__global__ void seg_dh0_kernel(const int32_t* __restrict__ plan, const int32_t* __restrict__ seg_seq, int nmax,
                               int Hv, int64_t state, const float* __restrict__ dh0_seg,
                               const float* __restrict__ dh_final, float* __restrict__ dh0) {
    if (plan[0] != 0) return;
    const int n = blockIdx.x, hv = blockIdx.y;
    int j0, j1;
    seq_segments(seg_seq, nmax, n, j0, j1);
    float* d = dh0 + ((int64_t)n * Hv + hv) * state;
    const float* s = j1 > j0 ? dh0_seg + ((int64_t)j0 * Hv + hv) * state
                             : (dh_final ? dh_final + ((int64_t)n * Hv + hv) * state : nullptr);
    for (int64_t e = threadIdx.x; e < state; e += blockDim.x) d[e] = s ? s[e] : 0.f;
}

template <int DK>
gdn_status merge_dv(bool fwd, int dv, const int32_t* plan, const int32_t* seg_seq, int nmax, int num_seqs, int Hv,
                    const float* M, const float* NB, const float* init, float* out, cudaStream_t s) {
    const dim3 grid(num_seqs, Hv, dv / kTile);
#define GDN_MERGE(DV)                                                                                       \
    if (fwd) seg_merge_fwd_kernel<DK, DV><<<grid, kMergeThreads, 0, s>>>(plan, seg_seq, nmax, Hv, M, NB, init, out); \
    else seg_merge_bwd_kernel<DK, DV><<<grid, kMergeThreads, 0, s>>>(plan, seg_seq, nmax, Hv, M, NB, init, out);
    switch (dv) {
        case 32: GDN_MERGE(32) break;
        case 64: GDN_MERGE(64) break;
        case 128: GDN_MERGE(128) break;
        default: return fail(GDN_ERR_UNSUPPORTED_SHAPE, "merge: dv must be 32, 64 or 128");
    }
#undef GDN_MERGE
    return check_launch(fwd ? "seg_merge_fwd_kernel" : "seg_merge_bwd_kernel");
}

}  // namespace

gdn_status launch_segments(const int32_t* plan, int num_seqs, int P, int T, int nmax, int32_t* cu_seg,
                           int32_t* seg_seq, cudaStream_t s) {
    segments_kernel<<<P < 148 ? P : 148, 128, 0, s>>>(plan, num_seqs, P, T, nmax, cu_seg, seg_seq);
    return check_launch("segments_kernel");
}

gdn_status launch_seg_merge(bool fwd, const int32_t* plan, const int32_t* seg_seq, int nmax, int num_seqs, int Hv,
                            int dk, int dv, const float* M, const float* NB, const float* init, float* out,
                            cudaStream_t s) {
    switch (dk) {
        case 32: return merge_dv<32>(fwd, dv, plan, seg_seq, nmax, num_seqs, Hv, M, NB, init, out, s);
        case 64: return merge_dv<64>(fwd, dv, plan, seg_seq, nmax, num_seqs, Hv, M, NB, init, out, s);
        case 128: return merge_dv<128>(fwd, dv, plan, seg_seq, nmax, num_seqs, Hv, M, NB, init, out, s);
    }
    return fail(GDN_ERR_UNSUPPORTED_SHAPE, "merge: dk must be 32, 64 or 128");
}

gdn_status launch_seg_dh0(const int32_t* plan, const int32_t* seg_seq, int nmax, int num_seqs, int Hv, int dk,
                          int dv, const float* dh0_seg, const float* dh_final, float* dh0, cudaStream_t s) {
    seg_dh0_kernel<<<dim3(num_seqs, Hv), 256, 0, s>>>(plan, seg_seq, nmax, Hv, (int64_t)dk * dv, dh0_seg, dh_final,
                                                       dh0);
    return check_launch("seg_dh0_kernel");
}

}  // namespace gdn
