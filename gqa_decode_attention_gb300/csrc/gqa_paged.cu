// gqa_paged.cu -- sparse paged FP8 decode kernel and its test hooks.
#include "gqa_launch.h"
#include "gqa_paged_kernel.cuh"

namespace gqa {

template <int D, int NT, int HB>
static cudaError_t launch_paged_inst(const PagedArgs &a, cudaStream_t stream) {
    using C = PagedCfg<D, NT, HB>;
    auto kern = gqa_paged_fp8_kernel<D, NT, HB>;
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    // Programmatic dependent launch: the CTAs may be scheduled while the
    // previous kernel in the stream drains; they wait for it before reading.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((a.Hkv + HB - 1) / HB, a.B);
    cfg.blockDim = dim3(C::THREADS);
    cfg.dynamicSmemBytes = C::SMEM_BYTES;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, a);
}

// Heads per CTA: the smallest power of two covering the KV heads, at most 8
// (4 when each consumer holds two n-tiles of query rows).
template <int D, int NT>
static cudaError_t launch_paged_nt(const PagedArgs &a, cudaStream_t stream) {
    const int cap = NT == 2 ? 4 : 8;
    const int want = a.Hkv < cap ? a.Hkv : cap;
    if (want <= 1) return launch_paged_inst<D, NT, 1>(a, stream);
    if (want <= 2) return launch_paged_inst<D, NT, 2>(a, stream);
    if (want <= 4 || NT == 2) return launch_paged_inst<D, NT, 4>(a, stream);
    return launch_paged_inst<D, NT, (NT == 2 ? 4 : 8)>(a, stream);
}

cudaError_t launch_paged_fp8(const PagedArgs &a, int D, cudaStream_t stream) {
    const bool two = a.G > 8;  // groups of 9..16 rows use two n-tiles of 8 rows
    if (D == 64) return two ? launch_paged_nt<64, 2>(a, stream) : launch_paged_nt<64, 1>(a, stream);
    if (D == 128) return two ? launch_paged_nt<128, 2>(a, stream) : launch_paged_nt<128, 1>(a, stream);
    return cudaErrorInvalidValue;
}

cudaError_t launch_paged_gather(const uint8_t *pool, const int32_t *page_table, const int32_t *topk, uint8_t *out,
                                int B, int Hkv, int D, int page_size, int pages_per_req, int num_pages, int topk_n,
                                unsigned *err, cudaStream_t stream) {
    const int n16 = Hkv * D / 16;
    const int threads = n16 < 256 ? ((n16 + 31) / 32) * 32 : 256;
    gqa_paged_gather_kernel<<<dim3(topk_n, B), threads, 0, stream>>>(pool, page_table, topk, out, Hkv, D, page_size,
                                                                     pages_per_req, num_pages, topk_n, err);
    return cudaGetLastError();
}

cudaError_t launch_fp8_to_f32(const uint8_t *codes, float *out, int n, cudaStream_t stream) {
    const int pairs = (n + 1) / 2;
    gqa_fp8_to_f32_kernel<<<(pairs + 255) / 256, 256, 0, stream>>>(codes, out, n);
    return cudaGetLastError();
}

}  // namespace gqa
