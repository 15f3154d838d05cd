// gqa_dense_impl.cuh -- launch templates of the dense split and combine kernels,
// instantiated by one translation unit per head size (d64, d128, d256, d192x128).
#pragma once

#include "gqa_dense_kernel.cuh"
#include "gqa_dense_umma.cuh"
#include "gqa_launch.h"

namespace gqa {

// D: score head size (q, K); DV: value head size (V, O).
template <int D, int DV, int CFG>
struct DenseInst {
    static constexpr int RB = 1 << CFG;
    static constexpr int T = dense_tile_keys(D, CFG);
    static constexpr int S = dense_stages(D, CFG);
    using C = DenseCfg<D, DV, RB, T, S>;
    static constexpr auto kernel() { return gqa_dense_split_kernel<D, DV, RB, T, S>; }
};

// The launches below rely on the kernel's dynamic shared-memory limit having
// been raised on the current device: the front end's occupancy query (once
// per device and kernel, under its lock) does that before any call launches.
// Key-lane instance CFG (0-3): dense_lane_lanes(CFG) key lanes of RB warps.
template <int D, int DV, int CFG>
struct DenseLaneInst {
    static constexpr int RB = 1 << dense_lane_rows_cfg(CFG);
    static constexpr int KS = dense_lane_lanes(CFG);
    static constexpr int T = dense_lane_tile_keys(D);
    static constexpr int S = dense_lane_stages(D, DV, CFG);
    using C = DenseCfg<D, DV, RB, T, S, KS>;
    static constexpr auto kernel() { return gqa_dense_split_kernel<D, DV, RB, T, S, KS>; }
};

template <int D, int DV, int CFG, template <int, int, int> class Inst = DenseInst>
static cudaError_t launch_split_cfg(const DenseLaunch &L) {
    using I = Inst<D, DV, CFG>;
    using C = typename I::C;
    auto kern = I::kernel();
    CUtensorMap tk, tv;
    if (!make_kv_tensor_map(&tk, L.k, L.args.B, L.args.Skv, L.args.Hkv, D, I::T) ||
        !make_kv_tensor_map(&tv, L.v, L.args.B, L.args.Skv, L.args.Hkv, DV, I::T))
        return cudaErrorInvalidValue;
    const dim3 grid(L.args.Hkv * L.args.row_groups, L.args.num_splits, L.args.B);
    const bool timed = L.ev_before != nullptr && L.ev_after != nullptr;
    if (timed) cudaEventRecord(L.ev_before, L.stream);
    kern<<<grid, C::THREADS, C::SMEM_BYTES, L.stream>>>(tk, tv, L.args);
    if (timed) cudaEventRecord(L.ev_after, L.stream);
    return cudaGetLastError();
}

template <int D, int DV, int CFG, template <int, int, int> class Inst = DenseInst>
static int occupancy_cfg() {
    using I = Inst<D, DV, CFG>;
    using C = typename I::C;
    auto kern = I::kernel();
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES) != cudaSuccess)
        return 0;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, C::THREADS, C::SMEM_BYTES) != cudaSuccess) return 0;
    return n;
}

template <int D>
static cudaError_t launch_combine(const DenseLaunch &L) {
    const DenseArgs &a = L.args;
    const long rows = long(a.B) * a.Hkv * a.Mq;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(rows));
    cfg.blockDim = dim3(kCombineThreads);
    cfg.dynamicSmemBytes = (size_t(combine_staged_splits<D>(a.num_splits)) * (D / 4) + kCombineThreads) * sizeof(float4);
    cfg.stream = L.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, gqa_combine_kernel<D>, (const float *)a.o_part, (const float *)a.lse_part,
                              a.out, a.lse, a.Sq, a.Hq, a.Hkv, a.G, a.Mq, a.num_splits);
}

// tcgen05 engine: one instance per head dim, 128 rows per CTA.
template <int D>
static cudaError_t launch_umma(const DenseLaunch &L) {
    using C = UmmaCfg<D>;
    auto kern = gqa_dense_umma_kernel<D>;
    CUtensorMap tk, tv;
    if (!make_kv_tensor_map(&tk, L.k, L.args.B, L.args.Skv, L.args.Hkv, D, C::BN) ||
        !make_kv_tensor_map(&tv, L.v, L.args.B, L.args.Skv, L.args.Hkv, D, C::BN))
        return cudaErrorInvalidValue;
    const dim3 grid(L.args.Hkv * L.args.row_groups, L.args.num_splits, L.args.B);
    const bool timed = L.ev_before != nullptr && L.ev_after != nullptr;
    if (timed) cudaEventRecord(L.ev_before, L.stream);
    kern<<<grid, C::THREADS, C::SMEM_BYTES, L.stream>>>(tk, tv, L.args);
    if (timed) cudaEventRecord(L.ev_after, L.stream);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess || L.args.num_splits == 1) return e;
    return launch_combine<D>(L);
}

template <int D>
static int umma_occupancy() {
    using C = UmmaCfg<D>;
    auto kern = gqa_dense_umma_kernel<D>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES) != cudaSuccess)
        return 0;
    return tmem_kernel_ctas_per_sm(reinterpret_cast<const void *>(kern), C::SMEM_BYTES, C::THREADS,
                                   int(C::TMEM_COLS));
}

template <int D, int DV = D>
static cudaError_t launch_dense(const DenseLaunch &L) {
    cudaError_t e;
    switch (L.cfg) {
        case 0: e = launch_split_cfg<D, DV, 0>(L); break;
        case 1: e = launch_split_cfg<D, DV, 1>(L); break;
        case 2: e = launch_split_cfg<D, DV, 2>(L); break;
        case 3: e = launch_split_cfg<D, DV, 3>(L); break;
        default:
            if constexpr (dense_has_lanes(D, DV)) {
                e = L.cfg == kLaneCfg       ? launch_split_cfg<D, DV, 0, DenseLaneInst>(L)
                    : L.cfg == kLaneCfg + 1 ? launch_split_cfg<D, DV, 1, DenseLaneInst>(L)
                    : L.cfg == kLaneCfg + 2 ? launch_split_cfg<D, DV, 2, DenseLaneInst>(L)
                                            : launch_split_cfg<D, DV, 3, DenseLaneInst>(L);
            } else {
                e = cudaErrorInvalidValue;
            }
            break;
    }
    if (e != cudaSuccess || L.args.num_splits == 1) return e;
    return launch_combine<DV>(L);
}

template <int D, int DV = D>
static int dense_occupancy(int cfg) {
    switch (cfg) {
        case 0: return occupancy_cfg<D, DV, 0>();
        case 1: return occupancy_cfg<D, DV, 1>();
        case 2: return occupancy_cfg<D, DV, 2>();
        case 3: return occupancy_cfg<D, DV, 3>();
        default:
            if constexpr (dense_has_lanes(D, DV)) {
                return cfg == kLaneCfg       ? occupancy_cfg<D, DV, 0, DenseLaneInst>()
                       : cfg == kLaneCfg + 1 ? occupancy_cfg<D, DV, 1, DenseLaneInst>()
                       : cfg == kLaneCfg + 2 ? occupancy_cfg<D, DV, 2, DenseLaneInst>()
                                             : occupancy_cfg<D, DV, 3, DenseLaneInst>();
            } else {
                return 0;
            }
    }
}

}  // namespace gqa
