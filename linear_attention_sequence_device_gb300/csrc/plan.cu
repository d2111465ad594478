// Shard plan on the device (flash-linear-attention page fla/ops/cp/context.py,
// get_cp_cu_seqlens steps 3-5): two binary searches per shard, the clamped
// slice of cu_seqlens compacted with a warp ballot (unique_consecutive), and
// the first/last-rank metadata.  One CTA; warp w handles shards w, w+W, ...
// No device-to-host copy of cu_seqlens is ever made.
#include "gdn_internal.cuh"

namespace gdn {
namespace {

constexpr int NT = 256;

// number of a[0..n) with a[i] <= x (a non-decreasing)
__device__ int count_le(const int32_t* a, int n, int x) {
    int lo = 0, hi = n;
    while (lo < hi) {
        int mid = (lo + hi) >> 1;
        if (a[mid] <= x) lo = mid + 1; else hi = mid;
    }
    return lo;
}
// number of a[0..n) with a[i] < x
__device__ int count_lt(const int32_t* a, int n, int x) {
    int lo = 0, hi = n;
    while (lo < hi) {
        int mid = (lo + hi) >> 1;
        if (a[mid] < x) lo = mid + 1; else hi = mid;
    }
    return lo;
}

__global__ void __launch_bounds__(NT) plan_kernel(const int32_t* __restrict__ cu, int N, int P,
                                                  int32_t* __restrict__ plan) {
    __shared__ int bad;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) bad = 0;
    __syncthreads();
    // validation: cu[0] == 0, non-decreasing, total divisible by P and >= P
    int my_bad = 0;
    if (tid == 0) {
        const int total = cu[N];
        my_bad = (cu[0] != 0) || (total < P) || (total % P != 0);
    }
    for (int i = tid; i < N; i += NT) my_bad |= (cu[i] > cu[i + 1]);
    if (my_bad) atomicOr(&bad, 1);
    __syncthreads();
    if (bad) {
        if (tid == 0) plan[0] = GDN_ERR_BAD_CU_SEQLENS;
        return;
    }
    const int total = cu[N];
    const int part = total / P;
    for (int r = warp; r < P; r += NT / 32) {
        const int rs = r * part, re = rs + part;
        const int s = count_le(cu + 1, N, rs);   // first sequence whose end > rs
        const int e = count_lt(cu, N, re);       // first sequence whose start >= re
        int32_t* lc = plan + GDN_PLAN_CU(N, P, r);
        int32_t* sq = plan + GDN_PLAN_SEQ(N, P, r);
        int count = 0;
        for (int base = s; base <= e; base += 32) {
            const int i = base + lane;
            const bool ok = i <= e;
            int c = 0, cp = -1;
            if (ok) {
                c = min(max(cu[i], rs), re) - rs;
                if (i > s) cp = min(max(cu[i - 1], rs), re) - rs;
            }
            const bool keep = ok && (i == s || c != cp);
            const unsigned m = __ballot_sync(0xffffffffu, keep);
            if (keep) {
                // a kept boundary is the first of its value, so the segment
                // that ends there belongs to the sequence just before it
                const int pos = count + __popc(m & ((1u << lane) - 1u));
                lc[pos] = c;
                if (pos > 0) sq[pos - 1] = i - 1;
            }
            count += __popc(m);
        }
        if (lane == 0) {
            int32_t* rec = plan + GDN_PLAN_REC(r);
            const int first_start = cu[s];
            const int last_end = cu[e];
            const int fr = first_start / part;
            const int lr = (last_end - 1) / part;
            rec[GDN_PLAN_LOCAL_NUM_SEQS] = count - 1;
            rec[GDN_PLAN_START_SEQ_IDX] = s;
            rec[GDN_PLAN_END_SEQ_IDX] = e;
            rec[GDN_PLAN_PRE_NUM_RANKS] = r - fr;
            rec[GDN_PLAN_POST_NUM_RANKS] = lr - r;
            rec[GDN_PLAN_IS_FIRST_RANK] = (r == fr);
            rec[GDN_PLAN_IS_LAST_RANK] = (r == lr);
            rec[GDN_PLAN_PRE_NUM_CONV_TOKENS] = max(0, rs - first_start);
        }
    }
    __syncthreads();
    // exclusive prefix sum of local_num_seqs -> SEG_OFFSET (warp 0)
    if (warp == 0) {
        int carry = 0;
        for (int base = 0; base < P; base += 32) {
            const int r = base + lane;
            int x = r < P ? plan[GDN_PLAN_REC(r) + GDN_PLAN_LOCAL_NUM_SEQS] : 0;
            int incl = x;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                int t = __shfl_up_sync(0xffffffffu, incl, off);
                if (lane >= off) incl += t;
            }
            if (r < P) plan[GDN_PLAN_REC(r) + GDN_PLAN_SEG_OFFSET] = carry + incl - x;
            carry += __shfl_sync(0xffffffffu, incl, 31);
        }
        if (lane == 0) plan[0] = 0;
    }
}

}  // namespace

gdn_status launch_plan(const int32_t* cu, int num_seqs, int P, int32_t* plan, cudaStream_t s) {
    plan_kernel<<<1, NT, 0, s>>>(cu, num_seqs, P, plan);
    return check_launch("plan_kernel");
}

}  // namespace gdn
