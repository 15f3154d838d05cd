// gqa_dense_d256.cu -- dense split-KV decode (and its combine), head dim 256.
#include "gqa_dense_impl.cuh"

namespace gqa {
// Head dim 256 runs on the tcgen05 engine for every group size (one engine per
// head dim keeps a row's arithmetic independent of the group size).
cudaError_t launch_dense_d256(const DenseLaunch &L) { return launch_umma<256>(L); }
int dense_ctas_per_sm_d256(int) { return umma_occupancy<256>(); }
}  // namespace gqa
