// gqa_paged.cu -- sparse paged FP8 decode kernel and its test hooks.
#include "gqa_launch.h"
#include "gqa_paged_kernel.cuh"

namespace gqa {

cudaError_t launch_paged_fp8(const PagedArgs &a, int D, cudaStream_t stream) {
    const dim3 grid((a.Hkv + kPagedHeadsPerCta - 1) / kPagedHeadsPerCta, a.B);
    const dim3 block(32 * kPagedHeadsPerCta);
    if (D == 64)
        gqa_paged_fp8_kernel<64><<<grid, block, 0, stream>>>(a);
    else if (D == 128)
        gqa_paged_fp8_kernel<128><<<grid, block, 0, stream>>>(a);
    else
        return cudaErrorInvalidValue;
    return cudaGetLastError();
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
