// gqa_dense_d64.cu -- dense split-KV decode and combine kernels, head dim 64.
#include "gqa_dense_impl.cuh"

namespace gqa {
cudaError_t launch_dense_d64(const DenseLaunch &L) { return launch_dense<64>(L); }
int dense_ctas_per_sm_d64(int cfg) { return dense_occupancy<64>(cfg); }
cudaError_t launch_combine_d64(const float *o_part, const float *lse_part, __nv_bfloat16 *out, float *lse, int B,
                              int Sq, int Hq, int Hkv, int G, int Mq, int S, cudaStream_t stream) {
    return launch_combine_rows<64>(o_part, lse_part, out, lse, B, Sq, Hq, Hkv, G, Mq, S, stream);
}
}  // namespace gqa
