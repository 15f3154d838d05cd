// gqa_dense_d128.cu -- dense split-KV decode (and its combine), head dim 128.
#include "gqa_dense_impl.cuh"

namespace gqa {
cudaError_t launch_dense_d128(const DenseLaunch &L) { return launch_dense<128>(L); }
int dense_ctas_per_sm_d128(int cfg) { return dense_occupancy<128>(cfg); }
}  // namespace gqa
