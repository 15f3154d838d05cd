// gqa_dense_d64.cu -- dense split-KV decode (and its combine), head dim 64.
#include "gqa_dense_impl.cuh"

namespace gqa {
cudaError_t launch_dense_d64(const DenseLaunch &L) { return launch_dense<64>(L); }
int dense_ctas_per_sm_d64(int cfg) { return dense_occupancy<64>(cfg); }
}  // namespace gqa
