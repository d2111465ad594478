// Token-major <-> head-major re-layout of per-head rows (the Ulysses wrapper's
// seq-to-heads / heads-to-seq exchange of the hyper-parallel page, which on
// one device is a move of whole d-element rows): [T, H, d] with token stride
// ld <-> dense [H, T, d].  Each thread moves 16-byte pieces; consecutive
// threads cover consecutive pieces of the head-major side, so the head-major
// writes (or reads) are contiguous and the token-major side is read (or
// written) 2*d bytes per row at a time.
#include "gdn_internal.cuh"

namespace gdn {
namespace {

constexpr int NT = 256;

template <bool TO_HEADS>
__global__ void __launch_bounds__(NT) relayout_kernel(const unsigned char* __restrict__ src,
                                                      unsigned char* __restrict__ dst, int64_t T, int H,
                                                      int row_bytes, int64_t ld_bytes) {
    const int pieces = row_bytes >> 4;  // 16-byte pieces per row
    const int64_t total = (int64_t)H * T * pieces;
    for (int64_t i = (int64_t)blockIdx.x * NT + threadIdx.x; i < total; i += (int64_t)gridDim.x * NT) {
        const int c = (int)(i % pieces);
        const int64_t ht = i / pieces;  // h * T + t
        const int64_t h = ht / T, t = ht - h * T;
        const int64_t tok = t * ld_bytes + h * row_bytes + 16 * c;  // token-major side
        const int64_t hm = ht * row_bytes + 16 * c;                 // head-major side
        if (TO_HEADS)
            *reinterpret_cast<uint4*>(dst + hm) = __ldg(reinterpret_cast<const uint4*>(src + tok));
        else
            *reinterpret_cast<uint4*>(dst + tok) = __ldg(reinterpret_cast<const uint4*>(src + hm));
    }
}

}  // namespace

gdn_status launch_relayout(const void* src, void* dst, int64_t T, int H, int d, int64_t ld, gdn_dtype dt,
                           bool to_heads, cudaStream_t s) {
    const int es = dt == GDN_BF16 ? 2 : 4;
    const int row_bytes = d * es;
    const int64_t total = (int64_t)H * T * (row_bytes >> 4);
    if (total == 0) return GDN_OK;
    int sms = 0, dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int64_t want = (total + NT - 1) / NT;
    const unsigned blocks = (unsigned)(want < 8ll * (sms > 0 ? sms : 1) ? want : 8ll * (sms > 0 ? sms : 1));
    const unsigned char* a = static_cast<const unsigned char*>(src);
    unsigned char* b = static_cast<unsigned char*>(dst);
    if (to_heads) relayout_kernel<true><<<blocks, NT, 0, s>>>(a, b, T, H, row_bytes, ld * es);
    else relayout_kernel<false><<<blocks, NT, 0, s>>>(a, b, T, H, row_bytes, ld * es);
    return check_launch("relayout_kernel");
}

}  // namespace gdn
