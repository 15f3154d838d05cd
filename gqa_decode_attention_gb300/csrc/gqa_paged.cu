// gqa_paged.cu -- sparse paged FP8 decode kernel and its test hooks.
#include "gqa_launch.h"
#include "gqa_paged_kernel.cuh"

namespace gqa {

template <int D, int NT>
static cudaError_t launch_paged_inst(const PagedArgs &a, cudaStream_t stream) {
    using C = PagedCfg<D, NT>;
    auto kern = gqa_paged_fp8_kernel<D, NT>;
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    const dim3 grid((a.Hkv + kPagedHeadsPerCta - 1) / kPagedHeadsPerCta, a.B);
    kern<<<grid, 32 * kPagedHeadsPerCta, C::SMEM_BYTES, stream>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_paged_fp8(const PagedArgs &a, int D, cudaStream_t stream) {
    const bool two = a.G > 8;  // groups of 9..16 rows use two n-tiles of 8 rows
    if (D == 64) return two ? launch_paged_inst<64, 2>(a, stream) : launch_paged_inst<64, 1>(a, stream);
    if (D == 128) return two ? launch_paged_inst<128, 2>(a, stream) : launch_paged_inst<128, 1>(a, stream);
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
