// gqa_noalloc.cu -- the dense decode for callers that cannot allocate.
//
// Some callers of this library cannot call cudaMalloc or any allocator at
// decode time: code running under a strict memory budget that was fixed at
// start-up, real-time loops where an allocation could block or fail, and
// hosts that hand the library only the tensors it must read and write.  For
// them, gqa_decode_noalloc runs the same split-KV kernels as gqa_decode_ex but
// keeps the split partials in a fixed scratch array compiled into the library
// instead of a per-call workspace, and it allocates nothing.
#include <cstdint>
#include <mutex>

#include "../../include/gqa_decode.h"

namespace {

constexpr size_t kScratchBytes = size_t(GQA_NOALLOC_SCRATCH_BYTES);
constexpr int kMaxDevices = 64;

// The scratch itself: one copy on every device that loads the library, held
// until the process exits.  Host code must not use this name as an address.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

std::mutex g_mu;
void *g_scratch_addr[kMaxDevices];

// Device address of the scratch on the current device; resolved once per
// device (the first call on that device), with that device current.
void *scratch_address(int dev) {
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_scratch_addr[dev] == nullptr) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) {
            cudaGetLastError();
            return nullptr;
        }
        g_scratch_addr[dev] = p;
    }
    return g_scratch_addr[dev];
}

}  // namespace

extern "C" gqa_status gqa_decode_noalloc(const void *q, const void *k, const void *v, void *out, float *lse,
                                         int B, int Sq, int Skv, int Hq, int Hkv, int D, float scale,
                                         int num_splits, gqa_stream_t stream) {
    if (num_splits < 0) return GQA_ERR_INVALID_ARG;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return GQA_ERR_CUDA;
    }
    // Size check first: a problem whose partials do not fit is refused before
    // anything is launched.  (0 also comes back for invalid shapes, which
    // gqa_decode_ex then reports.)
    const size_t need = gqa_decode_workspace_bytes(B, Sq, Skv, Hq, Hkv, D, num_splits);
    if (need > kScratchBytes) return GQA_ERR_NO_MEMORY;
    void *scratch = scratch_address(dev);
    if (scratch == nullptr) return GQA_ERR_CUDA;
    return gqa_decode_ex(q, k, v, out, lse, B, Sq, Skv, Hq, Hkv, D, scale, num_splits, scratch, kScratchBytes,
                         stream);
}

extern "C" size_t gqa_decode_noalloc_scratch_bytes(void) { return kScratchBytes; }
