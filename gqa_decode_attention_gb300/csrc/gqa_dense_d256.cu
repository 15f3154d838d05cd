// gqa_dense_d256.cu -- dense split-KV decode and combine kernels, head dim 256.
#include "gqa_dense_impl.cuh"

namespace gqa {
cudaError_t launch_dense_d256(const DenseLaunch &L) { return launch_dense<256>(L); }
int dense_ctas_per_sm_d256(int cfg) { return dense_occupancy<256>(cfg); }
}  // namespace gqa
