// gqa_paged.cu -- sparse (top-K) paged FP8 decode kernel and its test hooks.
#include "gqa_paged_impl.cuh"

namespace gqa {

// Test hook: byte copy of the selected rows through the kernel's own index map.
__global__ void gqa_paged_gather_kernel(const uint8_t *pool, const int32_t *page_table, const int32_t *topk,
                                        uint8_t *out, int Hkv, int D, int page_size, int pages_per_req,
                                        int num_pages, int topk_n, unsigned *err) {
    const int k = blockIdx.x;
    const int b = blockIdx.y;
    bool bad = false;
    const int t = topk[size_t(b) * topk_n + k];
    const int row = paged_token_row(page_table, b, pages_per_req, page_size, num_pages, t, &bad);
    if (bad && threadIdx.x == 0) flag_error(err, kErrIndex);
    const int n16 = Hkv * D / 16;
    uint4 *dst = reinterpret_cast<uint4 *>(out + (size_t(b) * topk_n + k) * Hkv * D);
    for (int u = threadIdx.x; u < n16; u += blockDim.x) {
        uint4 v = make_uint4(0, 0, 0, 0);
        if (row >= 0) v = *reinterpret_cast<const uint4 *>(pool + size_t(row) * Hkv * D + size_t(u) * 16);
        dst[u] = v;
    }
}

// Test hook: the kernel's E4M3FN -> f16 widening, reported as fp32.
__global__ void gqa_fp8_to_f32_kernel(const uint8_t *codes, float *out, int n) {
    const int i = (blockIdx.x * blockDim.x + threadIdx.x) * 2;
    if (i >= n) return;
    const uint16_t two = uint16_t(codes[i]) | (i + 1 < n ? uint16_t(codes[i + 1]) << 8 : uint16_t(0));
    const uint32_t h2 = e4m3x2_to_f16x2(two);
    const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&h2));
    out[i] = f.x;
    if (i + 1 < n) out[i + 1] = f.y;
}


cudaError_t launch_paged_topk_fp8(const PagedArgs &a, int D, cudaStream_t stream) {
    return cudaError_t(paged_dispatch<kKvFp8, false>(a, D, stream, 0));
}
int paged_topk_ctas_per_sm_fp8(const PagedArgs &a, int D) { return int(paged_dispatch<kKvFp8, false>(a, D, nullptr, 1)); }
cudaError_t launch_paged_topk_combine_fp8(const PagedArgs &a, int D, cudaStream_t stream) {
    const int hb = paged_heads_per_cta(D, true, a.Mq, a.Hkv);
    return D == 64 ? launch_paged_combine<64>(a, hb, stream) : launch_paged_combine<128>(a, hb, stream);
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
