// gqa_dense_d192x128.cu -- dense split-KV decode with a score head size of 192
// and a value head size of 128 (the d192x128 flavour); the combine kernel is
// the head-size-128 one.
#include "gqa_dense_impl.cuh"

namespace gqa {
cudaError_t launch_dense_d192x128(const DenseLaunch &L) { return launch_dense<192, 128>(L); }
int dense_ctas_per_sm_d192x128(int cfg) { return dense_occupancy<192, 128>(cfg); }
}  // namespace gqa
