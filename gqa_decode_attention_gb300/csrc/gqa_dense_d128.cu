// gqa_dense_d128.cu -- dense split-KV decode and combine kernels, head dim 128.
#include "gqa_dense_impl.cuh"

namespace gqa {
cudaError_t launch_dense_d128(const DenseLaunch &L) { return launch_dense<128>(L); }
int dense_ctas_per_sm_d128(int cfg) { return dense_occupancy<128>(cfg); }
cudaError_t launch_combine_d128(const float *o_part, const float *lse_part, __nv_bfloat16 *out, float *lse, int B,
                              int Sq, int Hq, int Hkv, int G, int Mq, int S, cudaStream_t stream) {
    return launch_combine_rows<128>(o_part, lse_part, out, lse, B, Sq, Hq, Hkv, G, Mq, S, stream);
}
}  // namespace gqa
