// Work order of a ticket-scheduled chunk launch, computed once per launch.
//
// Items are the token ranges (sequence or shard segment) of a chunk launch;
// each item runs for every (value head, column tile) pair.  With C = 64 and
// T* = max(longest item, total chunks of all heads and tiles / SMs), an item
// of L chunks may be split into a first and a second part; the second part
// starts from the first's final state, handed over through a final-state
// destination (flagged per (item, head, tile) pair).  Two rules:
//  * halves (single-segment launches with final states): an item with
//    T*/2 < L < 0.7 T* is split in the middle, so that long items start at
//    once and their second halves fill the end of the launch;
//  * tail (shard passes): when the launch holds more jobs than SMs and its
//    items are of similar length (shortest >= half the longest), every item
//    of at least 2s chunks is split into L - s and s chunks, with
//    s = ceil(SMs * longest / (jobs + SMs)).  The short second parts come
//    last and even out the end of the launch, which whole jobs of equal
//    length would leave ragged (jobs / SMs is rarely a whole number).
// Entries (whole items, first and second parts) are ordered: long wholes and
// first parts by decreasing length, then short wholes and second parts by
// decreasing length, ties by item.  Every first part is thus handed out
// before any second part that waits on it.
//
// Layout of the schedule words (int32, device):
//   [0]                    ticket counter, zeroed here
//   [1]                    number of entries n
//   [2]                    status word, zeroed here (a chunk kernel whose bounded
//                          wait expires writes GDN_ERR_TIMEOUT into it)
//   [4, 4 + S*m)           hand-over flags, one per (item, head, tile), zeroed here
//   [o + 2r, o + 2r + 1]   entry of rank r < n: item | part << 16, chunks of the
//                          first part (o = 4 + S*m rounded up to even)
// part: 0 whole item, 1 first part, 2 second part.
#include "gdn_internal.cuh"

namespace gdn {
namespace {

constexpr int kOrderThreads = 1024;

__global__ void __launch_bounds__(kOrderThreads) order_kernel(const ChunkParams p, int src, int S, int m,
                                                            int split_rule) {
    __shared__ int len[kMaxLptItems];
    __shared__ unsigned long long key[2 * kMaxLptItems];
    __shared__ int s_max, s_min, s_items, s_n;
    __shared__ unsigned long long s_sum;
    const int tid = threadIdx.x;
    int32_t* const w = p.sched;
    if (tid == 0) {
        s_max = 0;
        s_min = 0x7fffffff;
        s_items = 0;
        s_sum = 0ull;
        s_n = 0;
    }
    for (int64_t i = tid; i < (int64_t)S * m; i += kOrderThreads) w[kSchedHeader + i] = 0;
    __syncthreads();
    const int nvt = p.dv / p.col_tile;
    for (int x = tid; x < S; x += kOrderThreads) {
        const int l = job_item_length(p, src, x);
        const int c = l > 0 ? (l + 63) / 64 : 0;
        len[x] = c;
        atomicMax(&s_max, c);
        if (c > 0) {
            atomicMin(&s_min, c);
            atomicAdd(&s_items, 1);
        }
        atomicAdd(&s_sum, (unsigned long long)c * (unsigned long long)(p.Hv * nvt));
    }
    __syncthreads();
    const int sms = p.num_sms > 0 ? p.num_sms : 1;
    const long long avg = (long long)((s_sum + sms - 1) / sms);
    const int tstar = (int)(avg > s_max ? avg : s_max);
    // tail rule: the second parts' length s (0: no split)
    int tail = 0;
    if (split_rule == kSplitTail) {
        const long long jobs = (long long)s_items * p.Hv * nvt;
        if (jobs > sms && s_max >= 8 && 2 * s_min >= s_max)
            tail = (int)(((long long)sms * s_max + jobs + sms - 1) / (jobs + sms));
    }
    // chunks of the first part of an item of L chunks (0: whole)
    auto split_at = [&](int L) -> int {
        if (split_rule == kSplitHalves) return (L >= 2 && 2 * L > tstar && 10 * L < 7 * tstar) ? (L + 1) / 2 : 0;
        if (tail > 0 && L >= 2 * tail) return L - tail;
        return 0;
    };
    // key of entry e = 2x + h: group (bit 40), (2^30 - 1 - length) << 10, e
    int N2 = 1;
    while (N2 < 2 * S) N2 <<= 1;
    for (int e = tid; e < N2; e += kOrderThreads) {
        unsigned long long k = ~0ull;  // no entry: sorts last
        if (e < 2 * S) {
            const int x = e >> 1, h = e & 1, L = len[x];
            int grp = -1, el = 0;
            const int a = split_at(L);
            if (a > 0) {
                el = h ? L - a : a;
                grp = h;
            } else if (!h) {
                el = L;
                grp = 2 * L > tstar ? 0 : 1;
            }
            if (grp >= 0)
                k = ((unsigned long long)grp << 40) |
                    ((unsigned long long)((1u << 30) - 1u - (unsigned)el) << 10) | (unsigned long long)e;
        }
        key[e] = k;
    }
    __syncthreads();
    // bitonic sort, ascending
    for (int size = 2; size <= N2; size <<= 1) {
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            for (int i = tid; i < N2 / 2; i += kOrderThreads) {
                const int lo = 2 * i - (i & (stride - 1)), hi = lo + stride;
                const bool up = (lo & size) == 0;
                const unsigned long long a = key[lo], b = key[hi];
                if ((a > b) == up) {
                    key[lo] = b;
                    key[hi] = a;
                }
            }
            __syncthreads();
        }
    }
    int32_t* const order = w + chunk_sched_order_off(S, m);
    for (int r = tid; r < N2; r += kOrderThreads) {
        const unsigned long long k = key[r];
        if (k == ~0ull) continue;
        const int e = (int)(k & 1023u), x = e >> 1, L = len[x];
        const int a = split_at(L);
        const int part = a > 0 ? 1 + (e & 1) : 0;
        order[2 * r] = x | (part << 16);
        order[2 * r + 1] = a;
        atomicAdd(&s_n, 1);
    }
    __syncthreads();
    if (tid == 0) {
        w[0] = 0;
        w[1] = s_n;
        w[2] = 0;
        w[3] = 0;
    }
}

}  // namespace

gdn_status launch_chunk_order(const ChunkParams& p, int src, int S, int m, int split_rule, cudaStream_t s) {
    if (S < 1 || S > kMaxLptItems) return GDN_ERR_INVALID_ARG;
    order_kernel<<<1, kOrderThreads, 0, s>>>(p, src, S, m, split_rule);
    return check_launch("order_kernel");
}

}  // namespace gdn
