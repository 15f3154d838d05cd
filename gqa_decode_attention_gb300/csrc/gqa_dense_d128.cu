// gqa_dense_d128.cu -- dense split-KV decode (and its combine), head dim 128:
// the mma.sync engine for calls with few decode rows per head, the tcgen05
// engine for calls with many (the slot kUmmaCfg).
#include "gqa_dense_impl.cuh"

namespace gqa {
cudaError_t launch_dense_d128(const DenseLaunch &L) {
    return L.cfg == kUmmaCfg ? launch_umma<128>(L) : launch_dense<128>(L);
}
int dense_ctas_per_sm_d128(int cfg) { return cfg == kUmmaCfg ? umma_occupancy<128>() : dense_occupancy<128>(cfg); }
}  // namespace gqa
