// gqa_paged_kv_fp8.cu -- paged decode over whole requests, FP8 E4M3FN pools.
#include "gqa_paged_impl.cuh"

namespace gqa {
cudaError_t launch_paged_range_fp8(const PagedArgs &a, int D, cudaStream_t stream) {
    return cudaError_t(paged_dispatch<kKvFp8, true>(a, D, stream, 0));
}
int paged_range_ctas_per_sm_fp8(const PagedArgs &a, int D) { return int(paged_dispatch<kKvFp8, true>(a, D, nullptr, 1)); }
cudaError_t launch_paged_range_combine_fp8(const PagedArgs &a, int D, cudaStream_t stream) {
    const int hb = paged_heads_per_cta(D, true, a.Mq, a.Hkv);
    return D == 64 ? launch_paged_combine<64>(a, hb, stream) : launch_paged_combine<128>(a, hb, stream);
}
}  // namespace gqa
