// gqa_paged_impl.cuh -- launch templates of the paged kernel and its merge
// pass, shared by the translation units that instantiate its forms (top-K
// FP8; whole-request bf16, FP8 and int8).
#pragma once

#include "gqa_launch.h"
#include "gqa_paged_kernel.cuh"

namespace gqa {

// The kernel's dynamic shared-memory limit is raised on each device by the
// front end's occupancy query (once per device and instance, under its lock),
// which every call makes before it launches.
template <int D, int NT, int HB, int KVT, bool RANGE>
static cudaError_t launch_paged_inst(const PagedArgs &a, cudaStream_t stream) {
    using C = PagedCfg<D, NT, HB, KVT != kKvBf16>;
    auto kern = gqa_paged_kernel<D, NT, HB, KVT, RANGE>;
    // Programmatic dependent launch: the CTAs may be scheduled while the
    // previous kernel in the stream drains; they wait for it before reading.
    cudaLaunchConfig_t cfg = {};
    // (head block, worker of the balanced schedule)
    cfg.gridDim = dim3((a.Hkv + HB - 1) / HB, a.num_splits, 1);
    cfg.blockDim = dim3(C::THREADS);
    cfg.dynamicSmemBytes = C::SMEM_BYTES;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, a);
}

template <int D, int NT, int HB, int KVT, bool RANGE>
static int paged_occupancy_inst() {
    using C = PagedCfg<D, NT, HB, KVT != kKvBf16>;
    auto kern = gqa_paged_kernel<D, NT, HB, KVT, RANGE>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES) != cudaSuccess)
        return 0;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, C::THREADS, C::SMEM_BYTES) != cudaSuccess) return 0;
    return n;
}

// Dispatch over (n-tiles, heads per CTA).  op 0 launches, op 1 returns the
// resident CTAs per SM of the chosen instance (as a cudaError_t-sized int).
template <int D, int NT, int KVT, bool RANGE>
static long paged_dispatch_nt(const PagedArgs &a, cudaStream_t stream, int op) {
    constexpr bool KV8 = KVT != kKvBf16;
    const int hb = paged_heads_per_cta(D, KV8, a.Mq, a.Hkv);
#define GQA_PAGED_CASE(HBV)                                                                              \
    if (hb == HBV)                                                                                       \
        return op == 0 ? long(launch_paged_inst<D, NT, HBV, KVT, RANGE>(a, stream))                      \
                       : long(paged_occupancy_inst<D, NT, HBV, KVT, RANGE>());
    GQA_PAGED_CASE(1)
    GQA_PAGED_CASE(2)
    GQA_PAGED_CASE(4)
    if constexpr (NT == 1 && (KV8 || D == 64)) {
        GQA_PAGED_CASE(8)
    }
#undef GQA_PAGED_CASE
    return op == 0 ? long(cudaErrorInvalidValue) : 0L;
}

// Merge of the shared requests' partials (whole-request form, several workers).
template <int D>
static cudaError_t launch_paged_combine(const PagedArgs &a, int hb, cudaStream_t stream) {
    // CTA (b, y): rows 8 y .. 8 y + 7 of request b
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(a.B), unsigned((a.Hkv * a.Mq + kPagedMergeRows - 1) / kPagedMergeRows));
    cfg.blockDim = dim3(32 * kPagedMergeRows);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, gqa_paged_combine_kernel<D>, a, hb);
}

template <int KVT, bool RANGE>
static long paged_dispatch(const PagedArgs &a, int D, cudaStream_t stream, int op) {
    const bool two = a.Mq > 8;  // 9..16 rows use two n-tiles of 8 rows
    if (D == 64) return two ? paged_dispatch_nt<64, 2, KVT, RANGE>(a, stream, op) : paged_dispatch_nt<64, 1, KVT, RANGE>(a, stream, op);
    if (D == 128) return two ? paged_dispatch_nt<128, 2, KVT, RANGE>(a, stream, op) : paged_dispatch_nt<128, 1, KVT, RANGE>(a, stream, op);
    return op == 0 ? long(cudaErrorInvalidValue) : 0L;
}

}  // namespace gqa
