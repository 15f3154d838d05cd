// gqa_paged_umma.cu -- launchers of the paged decode on tcgen05 (FP8 pools,
// head dim 128, multiples of 8 KV heads, up to 4 query rows per KV head), for
// the sparse top-K form and the whole-request form.
#include "gqa_launch.h"
#include "gqa_paged_umma.cuh"

namespace gqa {

namespace {

template <int R, bool RANGE>
cudaError_t launch_inst(const PagedArgs &a, cudaStream_t stream) {
    using C = PagedUmmaCfg<R>;
    // (head block of 8 KV heads, worker of the balanced schedule); programmatic
    // dependent launch: the CTAs may start while the previous kernel drains.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(a.Hkv / C::HB), unsigned(a.num_splits), 1);
    cfg.blockDim = dim3(C::THREADS);
    cfg.dynamicSmemBytes = C::SMEM_BYTES;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, gqa_paged_umma_kernel<R, RANGE>, a);
}

// Resident CTAs per SM, from the kernel's own resource use: shared memory
// (with the per-CTA reservation), registers, threads and tensor-memory
// columns.  The runtime's occupancy query reports 1 for every kernel that
// allocates tensor memory, whatever it allocates, while the SM runs as many
// such CTAs as their columns fit (measured: 256 CTAs of 128 columns on 152
// SMs all start within 0.3 us).  Also raises the kernel's dynamic
// shared-memory limit on the current device.
template <int R, bool RANGE>
int occupancy_inst() {
    using C = PagedUmmaCfg<R>;
    auto kern = gqa_paged_umma_kernel<R, RANGE>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES) != cudaSuccess)
        return 0;
    return tmem_kernel_ctas_per_sm(reinterpret_cast<const void *>(kern), C::SMEM_BYTES, C::THREADS,
                                   int(C::TMEM_COLS));
}

}  // namespace

cudaError_t launch_paged_umma(const PagedArgs &a, bool range, cudaStream_t stream) {
    const int R = paged_umma_rows(a.Mq);
    if (range) return R == 2 ? launch_inst<2, true>(a, stream) : launch_inst<4, true>(a, stream);
    return R == 2 ? launch_inst<2, false>(a, stream) : launch_inst<4, false>(a, stream);
}

int paged_umma_ctas_per_sm(int Mq, bool range) {
    const int R = paged_umma_rows(Mq);
    if (range) return R == 2 ? occupancy_inst<2, true>() : occupancy_inst<4, true>();
    return R == 2 ? occupancy_inst<2, false>() : occupancy_inst<4, false>();
}

}  // namespace gqa
