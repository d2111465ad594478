// gdn_shard_fwd_noalloc: the sharded forward for callers that cannot
// allocate device memory themselves -- e.g. a plugin inside a host
// application that owns every device buffer and hands the plugin only its
// inputs and outputs, or a latency-critical loop that must not call
// cudaMalloc, which can synchronise the whole device.
//
// Its workspace is a fixed file-scope device array instead of a
// caller-provided buffer.  The array is created when the library's module is
// loaded on a device and lives until the process exits; its size bounds the
// problems this entry point accepts.
#include <mutex>

#include "gdn_internal.cuh"

namespace gdn {
namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[GDN_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
void* g_scratch_addr[kMaxDevices] = {};
void* g_scratch_ctx[kMaxDevices] = {};  // the context the cached address belongs to

typedef int (*CtxGetCurrentFn)(void**);

// The driver's cuCtxGetCurrent (through the runtime's entry-point query, so
// that the library needs no link against the driver library).
CtxGetCurrentFn ctx_get_current() {
    static CtxGetCurrentFn fn = nullptr;
    static bool tried = false;
    if (!tried) {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<CtxGetCurrentFn>(ptr);
        tried = true;
    }
    return fn;
}

// Device address of g_noalloc_scratch on the current device.  In host code
// the symbol is only a host-side stand-in, so the address is looked up with
// the device current and cached per device, together with the CUDA context
// it belongs to: a new primary context on the device (after cudaDeviceReset)
// reloads the module, and the address is looked up again.
gdn_status scratch_address(void** out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(GDN_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    if (dev < 0 || dev >= kMaxDevices)
        return fail(GDN_ERR_INVALID_ARG, "device %d beyond the %d supported", dev, kMaxDevices);
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    void* ctx = nullptr;
    CtxGetCurrentFn get = ctx_get_current();
    if (get) get(&ctx);
    if (!g_scratch_addr[dev] || g_scratch_ctx[dev] != ctx) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || !p)
            return fail(GDN_ERR_CUDA, "cudaGetSymbolAddress(scratch): %s", cudaGetErrorString(e));
        if (!get || !ctx) {  // the runtime has made a context current by now
            ctx = nullptr;
            if (get) get(&ctx);
        }
        g_scratch_addr[dev] = p;
        g_scratch_ctx[dev] = ctx;
    }
    *out = g_scratch_addr[dev];
    return GDN_OK;
}

}  // namespace
}  // namespace gdn

using namespace gdn;

extern "C" gdn_status gdn_shard_fwd_noalloc(const void* x, const void* conv_w, const void* conv_b,
                                            int32_t conv_k, const float* g, const void* beta,
                                            const float* h0, const int32_t* cu_seqlens,
                                            int32_t num_seqs, int32_t T, int32_t Hk, int32_t Hv,
                                            int32_t dk, int32_t dv, float scale, uint32_t flags,
                                            int32_t n_shards, gdn_dtype dtype, void* o,
                                            float* h_final, int32_t* plan_out, void* stream) {
    const size_t need = gdn::shard_fwd_workspace_min(T, num_seqs, n_shards, Hk, Hv, dk, dv, dtype);
    if (need == 0)
        return fail(GDN_ERR_INVALID_ARG, "invalid sizes (T=%d num_seqs=%d n_shards=%d)", T, num_seqs,
                    n_shards);
    if (need > (size_t)GDN_NOALLOC_SCRATCH_BYTES)
        return fail(GDN_ERR_WORKSPACE,
                    "problem needs %zu bytes of scratch; gdn_shard_fwd_noalloc has a fixed %zu-byte "
                    "scratch array (use gdn_shard_fwd with a caller workspace)",
                    need, (size_t)GDN_NOALLOC_SCRATCH_BYTES);
    void* scratch = nullptr;
    gdn_status st = scratch_address(&scratch);
    if (st != GDN_OK) return st;
    // gdn_shard_fwd writes every workspace word it later reads, so the
    // previous call's contents need no clearing.
    return gdn_shard_fwd(x, conv_w, conv_b, conv_k, g, beta, h0, cu_seqlens, num_seqs, T, Hk, Hv,
                         dk, dv, scale, flags, n_shards, dtype, scratch,
                         (size_t)GDN_NOALLOC_SCRATCH_BYTES, o, h_final, plan_out, stream);
}
