// gqa_read_stream.cu -- a read-only HBM stream, the measurement hook that
// gives the benchmark a read-only bandwidth figure beside the copy peak.
//
// A decode kernel only reads its K/V bytes, and a read-only stream has no
// write-back traffic, so it can run above a device-to-device copy's rate.
// This kernel reads a buffer once with 16-byte non-caching loads (eight in
// flight per thread, a grid of four 512-thread CTAs per SM) and folds the
// words into one XOR so the loads cannot be removed.
#include <cstdint>

#include "../../include/gqa_decode.h"
#include "../../include/gqa_decode_debug.h"
#include "gqa_common.cuh"

namespace {

__device__ __forceinline__ uint4 ld_stream(const uint4 *p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

constexpr int kThreads = 512;
constexpr int kUnroll = 8;

__global__ void __launch_bounds__(kThreads) gqa_read_stream_kernel(const uint4 *p, size_t n, unsigned *sink) {
    const size_t stride = size_t(gridDim.x) * kThreads;
    size_t i = size_t(blockIdx.x) * kThreads + threadIdx.x;
    uint32_t acc = 0;
    for (; i + (kUnroll - 1) * stride < n; i += kUnroll * stride) {
        uint4 v[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) v[u] = ld_stream(p + i + u * stride);
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) acc ^= v[u].x ^ v[u].y ^ v[u].z ^ v[u].w;
    }
    for (; i < n; i += stride) {
        const uint4 v = ld_stream(p + i);
        acc ^= v.x ^ v.y ^ v.z ^ v.w;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc ^= __shfl_xor_sync(0xffffffffu, acc, off);
    if ((threadIdx.x & 31) == 0) atomicXor(sink, acc);
}

}  // namespace

extern "C" gqa_status gqa_debug_read_stream(const void *buf, size_t bytes, unsigned *sink, gqa_stream_t stream) {
    if (buf == nullptr || sink == nullptr || bytes == 0 || bytes % 16 != 0) return GQA_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(buf) & 15u) != 0 || (reinterpret_cast<uintptr_t>(sink) & 3u) != 0)
        return GQA_ERR_ALIGNMENT;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
        cudaGetLastError();
        return GQA_ERR_CUDA;
    }
    gqa_read_stream_kernel<<<4 * sms, kThreads, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint4 *>(buf), bytes / 16, sink);
    return cudaGetLastError() == cudaSuccess ? GQA_OK : GQA_ERR_CUDA;
}
