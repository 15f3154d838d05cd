// gqa_paged_kv_bf16.cu -- paged decode over whole requests, bf16 pools.
#include "gqa_paged_impl.cuh"

namespace gqa {
cudaError_t launch_paged_range_bf16(const PagedArgs &a, int D, cudaStream_t stream) {
    return cudaError_t(paged_dispatch<false, true>(a, D, stream, 0));
}
int paged_range_ctas_per_sm_bf16(const PagedArgs &a, int D) { return int(paged_dispatch<false, true>(a, D, nullptr, 1)); }
}  // namespace gqa
