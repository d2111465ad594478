// Causal depthwise conv1d + SiLU with the previous shard's halo
// (hyper-parallel page, _causal_conv1d_with_cp_halo; zero history before a
// sequence start as implied by the varlen plan's pre_num_conv_tokens).
//
// HBM-bound stencil.  Each thread owns 8 consecutive channels (one 16-byte
// bf16 vector, two for fp32) of a strip of R rows and slides a register
// window of the last conv_k - 1 input rows down the strip, so every input
// element is read once (plus conv_k - 1 halo rows per strip).  A warp covers
// 256 contiguous channels of a row: fully coalesced 512-byte transactions.
// Input rows stream through a per-thread ring of NSTAGE batches of RB rows in
// shared memory, filled by cp.async: the bytes in flight are bounded by
// shared memory rather than registers, and since every thread only reads
// what it copied itself, no block-level synchronisation is needed.
// Grid: (channel blocks, strips per shard, shards), with the strip length
// chosen at launch so that all CTAs fit in one wave of resident blocks.
#include "chunk_common.cuh"

namespace gdn {
namespace {

constexpr int NT = 128;
constexpr int RB = 4;      // rows per batch
constexpr int NSTAGE = 4;  // batches in the shared-memory ring

struct ConvParams {
    const void* x; int64_t ldx;
    void* y; int64_t ldy;
    const void* w; const void* b;
    int T, C, Kc;
    const int32_t* cu; int num_seqs;   // explicit mode (plan == null)
    const void* halo; int halo_len;    // explicit mode
    const int32_t* plan; int P;        // shard mode
    int rows;                          // rows per strip (a multiple of RB)
};

template <typename T> struct Vec8;
template <> struct Vec8<__nv_bfloat16> {
    struct Raw { uint4 v; };  // eight bf16 as loaded
    static __device__ __forceinline__ Raw load_raw(const __nv_bfloat16* p) {
        return Raw{*reinterpret_cast<const uint4*>(p)};
    }
    static __device__ __forceinline__ void unpack(const Raw& r, float* f) {
        const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&r.v);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            float2 t = __bfloat1622float2(h[i]);
            f[2 * i] = t.x;
            f[2 * i + 1] = t.y;
        }
    }
    static __device__ __forceinline__ void load(const __nv_bfloat16* p, float* f) {
        uint4 raw = *reinterpret_cast<const uint4*>(p);
        const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&raw);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            float2 t = __bfloat1622float2(h[i]);
            f[2 * i] = t.x;
            f[2 * i + 1] = t.y;
        }
    }
    static __device__ __forceinline__ void store(__nv_bfloat16* p, const float* f) {
        uint4 raw;
        __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&raw);
#pragma unroll
        for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
        *reinterpret_cast<uint4*>(p) = raw;
    }
};
template <> struct Vec8<float> {
    struct Raw { float4 a, b; };
    static __device__ __forceinline__ Raw load_raw(const float* p) {
        return Raw{reinterpret_cast<const float4*>(p)[0], reinterpret_cast<const float4*>(p)[1]};
    }
    static __device__ __forceinline__ void unpack(const Raw& r, float* f) {
        f[0] = r.a.x; f[1] = r.a.y; f[2] = r.a.z; f[3] = r.a.w;
        f[4] = r.b.x; f[5] = r.b.y; f[6] = r.b.z; f[7] = r.b.w;
    }
    static __device__ __forceinline__ void load(const float* p, float* f) {
        float4 a = reinterpret_cast<const float4*>(p)[0], b = reinterpret_cast<const float4*>(p)[1];
        f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
        f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
    }
    static __device__ __forceinline__ void store(float* p, const float* f) {
        reinterpret_cast<float4*>(p)[0] = make_float4(f[0], f[1], f[2], f[3]);
        reinterpret_cast<float4*>(p)[1] = make_float4(f[4], f[5], f[6], f[7]);
    }
};

// silu(a) for a bf16 result: 0.5 a (1 + tanh(a / 2)), one hardware tanh (its
// error, about 5e-4, is far below bf16 rounding); for fp32 results
// a / (1 + e^-a), the exponent capped so that the fast divide stays in range
// (silu(a) ~ 0 below that).
template <typename T>
__device__ __forceinline__ float silu(float a);
template <>
__device__ __forceinline__ float silu<__nv_bfloat16>(float a) {
    float t;
    asm("tanh.approx.f32 %0, %1;" : "=f"(t) : "f"(0.5f * a));
    return 0.5f * a * (1.f + t);
}
template <>
__device__ __forceinline__ float silu<float>(float a) {
    return __fdividef(a, 1.f + __expf(fminf(-a, 80.f)));
}

template <typename T, int KC>
__global__ void __launch_bounds__(NT) conv_kernel(const ConvParams p) {
    const int c0 = (blockIdx.x * NT + threadIdx.x) * 8;
    if (c0 >= p.C) return;
    int part, rs;
    const int32_t* lc;   // local cu_seqlens of this shard
    int nloc;            // number of local sequences
    int hlen;            // rows of history before local row 0 for the first sequence
    if (p.plan) {
        if (p.plan[0] != 0) return;  // malformed cu_seqlens
        const int r = blockIdx.z;
        part = p.T / p.P;
        rs = r * part;
        const int32_t* rec = p.plan + GDN_PLAN_REC(r);
        lc = p.plan + GDN_PLAN_CU(p.num_seqs, p.P, r);
        nloc = rec[GDN_PLAN_LOCAL_NUM_SEQS];
        hlen = min(KC - 1, (int)rec[GDN_PLAN_PRE_NUM_CONV_TOKENS]);
    } else {
        part = p.T;
        rs = 0;
        lc = p.cu;
        nloc = p.num_seqs;
        hlen = p.halo_len;
    }
    const int lt0 = blockIdx.y * p.rows;
    if (lt0 >= part) return;
    const int lt1 = min(part, lt0 + p.rows);
    const T* __restrict__ x = static_cast<const T*>(p.x);
    T* __restrict__ y = static_cast<T*>(p.y);

    float wr[KC][8], br[8];
    {
        const T* w = static_cast<const T*>(p.w);
#pragma unroll
        for (int c = 0; c < 8; ++c) {
#pragma unroll
            for (int j = 0; j < KC; ++j) wr[j][c] = Elem<T>::to_f(w[(int64_t)(c0 + c) * KC + j]);
            br[c] = p.b ? Elem<T>::to_f(static_cast<const T*>(p.b)[c0 + c]) : 0.f;
        }
    }
    // local sequence containing row lt0 and the next boundary after it
    int seg = upper_bound_minus1(lc, nloc, lt0);
    if (seg > nloc - 1) seg = nloc - 1;  // lt0 == part cannot happen; guard anyway
    int seg_start = lc[seg];
    int next = seg + 1 <= nloc ? lc[seg + 1] : part;

    // window: win[j] holds input row (t - (KC-1) + j) for j < KC-1
    float win[KC > 1 ? KC - 1 : 1][8];
#pragma unroll
    for (int j = 0; j < KC - 1; ++j) {
        const int lrow = lt0 - (KC - 1) + j;  // local row index of the history entry
        bool have = false;
        const T* src = nullptr;
        if (lrow >= seg_start && lrow >= 0) {
            have = true;
            src = x + (int64_t)(rs + lrow) * p.ldx + c0;
        } else if (seg == 0 && seg_start - lrow <= hlen) {
            const int m = seg_start - lrow;  // rows before the shard start (1 = adjacent)
            have = true;
            if (p.plan) src = x + (int64_t)(rs - m) * p.ldx + c0;  // previous shard's rows
            else src = static_cast<const T*>(p.halo) + (int64_t)(KC - 1 - m) * p.C + c0;
        }
        if (have) Vec8<T>::load(src, win[j]);
        else {
#pragma unroll
            for (int c = 0; c < 8; ++c) win[j][c] = 0.f;
        }
    }
    // ring of NSTAGE batches: stage b holds rows [lt0 + RB b, lt0 + RB (b + 1))
    constexpr int VEC = sizeof(T) * 8 / 16;  // 16-byte vectors per row and thread
    extern __shared__ uint4 ring[];          // [NSTAGE][RB][VEC][NT]
    const int nb = (lt1 - lt0 + RB - 1) / RB;
    auto issue = [&](int b) {
        if (b < nb) {
            uint4* st = ring + (size_t)(b % NSTAGE) * RB * VEC * NT;
#pragma unroll
            for (int u = 0; u < RB; ++u) {
                const int t = lt0 + RB * b + u;
                const T* src = x + (int64_t)(rs + (t < lt1 ? t : lt0)) * p.ldx + c0;
#pragma unroll
                for (int v = 0; v < VEC; ++v)
                    cp_async16(st + (u * VEC + v) * NT + threadIdx.x, reinterpret_cast<const uint4*>(src) + v,
                               t < lt1 ? 16 : 0);
            }
        }
        cp_async_commit();
    };
#pragma unroll
    for (int b = 0; b < NSTAGE - 1; ++b) issue(b);
    for (int b = 0; b < nb; ++b) {
        issue(b + NSTAGE - 1);
        cp_async_wait<NSTAGE - 1>();
        const uint4* st = ring + (size_t)(b % NSTAGE) * RB * VEC * NT;
#pragma unroll
        for (int u = 0; u < RB; ++u) {
            const int t = lt0 + RB * b + u;
            if (t >= lt1) break;
            while (t == next) {  // a new sequence starts: no history
#pragma unroll
                for (int j = 0; j < KC - 1; ++j)
#pragma unroll
                    for (int c = 0; c < 8; ++c) win[j][c] = 0.f;
                ++seg;
                next = seg + 1 <= nloc ? lc[seg + 1] : part;
            }
            float cur[8], out[8];
            uint4 rv[VEC];
#pragma unroll
            for (int v = 0; v < VEC; ++v) rv[v] = st[(u * VEC + v) * NT + threadIdx.x];
            Vec8<T>::unpack(*reinterpret_cast<const typename Vec8<T>::Raw*>(rv), cur);
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                float acc = br[c];
#pragma unroll
                for (int j = 0; j < KC - 1; ++j) acc = fmaf(wr[j][c], win[j][c], acc);
                acc = fmaf(wr[KC - 1][c], cur[c], acc);
                out[c] = silu<T>(acc);
            }
            Vec8<T>::store(y + (int64_t)(rs + t) * p.ldy + c0, out);
#pragma unroll
            for (int j = 0; j + 1 < KC - 1; ++j)
#pragma unroll
                for (int c = 0; c < 8; ++c) win[j][c] = win[j + 1][c];
            if (KC > 1) {
#pragma unroll
                for (int c = 0; c < 8; ++c) win[KC > 1 ? KC - 2 : 0][c] = cur[c];
            }
        }
    }
}

}  // namespace

gdn_status set_smem_attr(const void* func, size_t bytes);

namespace {

// Resident CTAs of the instance on the current device (cached per device).
template <typename T, int KC>
int resident_slots(size_t smem) {
    static int cache[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    if (cache[dev] > 0) return cache[dev];
    int sms = 0, per = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, conv_kernel<T, KC>, NT, smem) != cudaSuccess)
        return 0;
    return cache[dev] = sms * per;
}

template <typename T, int KC>
gdn_status launch_tk(ConvParams p, dim3 grid, cudaStream_t s) {
    const size_t smem = (size_t)NSTAGE * RB * (sizeof(T) * 8 / 16) * NT * 16;
    gdn_status st = set_smem_attr((const void*)conv_kernel<T, KC>, smem);
    if (st != GDN_OK) return st;
    // strips per shard: the CTAs fill whole waves of resident slots (a partly
    // filled last wave moves its bytes at a fraction of the bandwidth), with
    // strips of at least 64 rows so that the K-1 halo rows stay a small overhead
    const int part = p.T / p.P;
    const int slots = resident_slots<T, KC>(smem);
    const int per = (int)grid.x * p.P;
    const int nmax = max(1, part / 64);
    int n = (part + 127) / 128;
    if (slots > 0) {
        n = 1;
        double best = 2.0;
        for (int c = 1; c <= nmax && c <= 1024; ++c) {
            const double waves = (double)per * c / slots, full = ceil(waves);
            const double idle = (full - waves) / full;  // share of the launched waves' slots left idle
            if (idle < best - 1e-9) {
                best = idle;
                n = c;
            }
            if (best < 0.02) break;
        }
    }
    n = min(n, nmax);
    int rows = (part + n - 1) / n;
    p.rows = (rows + RB - 1) / RB * RB;
    grid.y = (part + p.rows - 1) / p.rows;
    conv_kernel<T, KC><<<grid, NT, smem, s>>>(p);
    return check_launch("conv_kernel");
}

template <typename T>
gdn_status launch_t(const ConvParams& p, dim3 grid, cudaStream_t s) {
    switch (p.Kc) {
        case 1: return launch_tk<T, 1>(p, grid, s);
        case 2: return launch_tk<T, 2>(p, grid, s);
        case 3: return launch_tk<T, 3>(p, grid, s);
        case 4: return launch_tk<T, 4>(p, grid, s);
    }
    return fail(GDN_ERR_UNSUPPORTED_SHAPE, "conv_k=%d not in 1..4", p.Kc);
}

}  // namespace

gdn_status launch_conv(const void* x, int64_t ldx, gdn_dtype dt, int T, int C, const void* w,
                       const void* b, int Kc, const int32_t* cu, int num_seqs, const void* halo,
                       int halo_len, void* y, int64_t ldy, const int32_t* plan, int P,
                       cudaStream_t s) {
    ConvParams p{x, ldx, y, ldy, w, b, T, C, Kc, cu, num_seqs, halo, halo_len, plan, plan ? P : 1, 128};
    const int part = T / p.P;
    dim3 grid((C / 8 + NT - 1) / NT, 1, p.P);
    if (part <= 0) return GDN_OK;
    return dt == GDN_BF16 ? launch_t<__nv_bfloat16>(p, grid, s) : launch_t<float>(p, grid, s);
}

}  // namespace gdn
