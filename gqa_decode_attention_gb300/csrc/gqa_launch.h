// gqa_launch.h -- host-side launch plumbing shared by the kernel translation
// units and the C-ABI front end (gqa_api.cu).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "gqa_params.h"

namespace gqa {

// Dense kernel instances, by the number of query rows a CTA holds: cfg c has
// 2^c consumer warps of 16 rows (16, 32, 64, 128 rows).  The TMA tile (keys
// per ring slot) and the ring depth are chosen per (head dim, cfg) so that
// small-group CTAs stay small and several fit on one SM.
constexpr int kDenseCfgs = 4;
inline int dense_cfg_for_rows(int rows) { return rows <= 16 ? 0 : rows <= 32 ? 1 : rows <= 64 ? 2 : 3; }
inline int dense_cfg_rows(int cfg) { return 16 << cfg; }
// The tcgen05 engine takes the slot after the mma.sync configurations.  It
// serves head dim 256 at every size, and head dim 128 once a call has at least
// GQA_D128_UMMA_MIN_SQ decode rows per head: with the usual groups of 8 or more
// query heads a CTA then holds 64 or more rows, the score and output
// contractions stop fitting the legacy tensor pipe's latency budget, and the
// 128-lane TMEM tile pays (with small groups the tcgen05 kernel runs a few
// points below the mma.sync one).  The choice depends on Sq and the head dims
// only, never on the group size, so a query row gets the same arithmetic with
// native GQA as with K/V expanded per head.
constexpr int kUmmaCfg = kDenseCfgs;
#ifndef GQA_D128_UMMA_MIN_SQ
#define GQA_D128_UMMA_MIN_SQ 8
#endif
inline bool dense_uses_umma(int D, int Dv, int Sq) {
    return D == 256 || (D == 128 && Dv == 128 && Sq >= GQA_D128_UMMA_MIN_SQ);
}
// Key-lane instances of the mma.sync kernel (cfg kLaneCfg + c): a CTA whose
// consumer warps form key lanes of RB warps (16 rows each) that split its
// walk and merge in shared memory.  c = 0: 16 rows, 4 lanes, 8-stage ring
// (one split of a long walk: two stages a lane, so each lane's next tile
// loads while it computes); c = 1: 32 rows, 4 lanes, 12 stages; c = 2: 16
// rows, 6 lanes, 12 stages (a whole small cache in one CTA); c = 3: 64 rows,
// 2 lanes of 4 warps, 12 stages (both uses; d128 only).  Head dims 64
// and 128, tiles of 16 KiB (64 keys at d64, 32 at d128); the d192x128
// flavour, 32-key tiles of 20 KiB and 8 stages in every instance.
//  - A small cache (K and V of a (batch row, KV head, row group) unit within
//    GQA_LANE_MAX_UNIT_BYTES) that the automatic split count would split runs
//    as one CTA per unit: one launch, no combine pass.  Measured on GB300
//    (device time per call, L2 flushed): 1K keys at d64 or 512 at d128 went
//    from 13.0-16.1 us to 10.9-13.0 us; at 512 KiB a unit the one-CTA walk was
//    already 1-2 us slower than splits + combine.
//  - Past that, few units split across one wave of key-lane CTAs (the plan
//    is in the front end).
// Ring depth: 12 stages (192 KiB of loads outstanding on the SM) took the
// 1K-key d64 cache from 11.8 to 10.9 us against 8 stages, while 8 stages were
// 4 % faster on a 128K-key walk split 19 ways, and 12 stages up to 6 % slower
// when split walks fill every SM; halving the tile to keep 16 or 24 stages
// cost 2 us on the small cache and up to 50 % on long walks.  For split walks
// 4 lanes with two stages each beat 8 lanes with one (the 128K-key two-row
// decode 87.0 -> 85.1 us, batch 1 with 4K keys 15.4 -> 13.4 us, no shape
// slower); 6 lanes with 12 stages gained more on some shapes but lost 6 % at
// 152 CTAs.  For a whole small cache 6 lanes over 12 stages matched or beat 8
// (batch 4 with 400 keys 12.3 -> 10.3 us) and 4 lanes lost 1.3 us on the
// 1K-key d64 cache.
constexpr int kLaneCfg = kUmmaCfg + 1;
constexpr int kLaneCfgs = 4;
#ifndef GQA_LANE_MAX_UNIT_BYTES
#define GQA_LANE_MAX_UNIT_BYTES (256 * 1024)
#endif
inline bool dense_is_lane_cfg(int cfg) { return cfg >= kLaneCfg && cfg < kLaneCfg + kLaneCfgs; }
// mma.sync row configuration (0: 16 rows, 1: 32, 2: 64) of key-lane instance c
// Key-lane instance for a CTA of mma.sync row configuration rc (0-2): a
// whole small cache (whole) or one split of a longer walk.
inline int dense_lane_cfg_for(int rc, bool whole) { return kLaneCfg + (rc == 2 ? 3 : rc == 1 ? 1 : whole ? 2 : 0); }
// Row configurations with key-lane instances in use: 16 and 32 rows, and 64
// rows at d128 (measured on GB300 with 64 rows a CTA: 64/4 heads at Sq 4 over
// 128K keys 94.3 -> 76.8 us, 128/8 heads at Sq 4, batch 2, 32K keys 101.4 ->
// 80.9 us; at d64 64/8 heads at Sq 8 over 64K keys went 48.2 -> 52.3 us, so
// d64 keeps the general choice there).
inline int dense_lane_row_cfgs(int D, int Dv) { return D == 128 && Dv == 128 ? 3 : 2; }
constexpr int dense_lane_rows_cfg(int c) { return c == 1 ? 1 : c == 3 ? 2 : 0; }
constexpr int dense_lane_tile_keys(int D) { return D == 64 ? 64 : 32; }
// (The d192x128 flavour's 20 KiB stages take 8 in every instance.)
constexpr int dense_lane_stages(int D, int DV, int c) { return c == 0 || D + DV > 256 ? 8 : 12; }
constexpr int dense_lane_lanes(int c) { return c == 2 ? 6 : c == 3 ? 2 : 4; }
// Head sizes with key-lane instances: 64 and 128 (D == Dv), and d192x128.
constexpr bool dense_has_lanes(int D, int DV) { return (D == DV && (D == 64 || D == 128)) || (D == 192 && DV == 128); }
// Query rows per CTA: the tcgen05 engine always holds 128 rows (its TMEM
// lanes); the mma.sync engine holds the group's rows rounded up to 16, at
// most 128 (16 or 32 in a key-lane instance).
inline int dense_rows_per_cta(int cfg) {
    return cfg == kUmmaCfg                ? 128
           : dense_is_lane_cfg(cfg) ? dense_cfg_rows(dense_lane_rows_cfg(cfg - kLaneCfg))
                                          : dense_cfg_rows(cfg);
}
// Tile keys and ring depth of the 16-row instance at D = 128 (the decode
// shape with the most traffic); compile-time knobs for tuning builds.
#ifndef GQA_D128_R16_TILE
#define GQA_D128_R16_TILE 16
#endif
#ifndef GQA_D128_R16_STAGES
#define GQA_D128_R16_STAGES 3
#endif
// (D is the score head size; the d192x128 flavour uses the D = 192 row.)
constexpr int dense_tile_keys(int D, int cfg) {
    return D == 64 ? (cfg == 0 ? 32 : 64) : D == 128 ? (cfg == 0 ? GQA_D128_R16_TILE : cfg == 1 ? 32 : 64)
         : D == 192 ? (cfg <= 1 ? 16 : 32)
                    : (cfg <= 1 ? 16 : cfg == 2 ? 32 : 64);
}
constexpr int dense_stages(int D, int cfg) {
    return D == 64 ? (cfg <= 1 ? 3 : 4) : D == 128 ? (cfg == 0 ? GQA_D128_R16_STAGES : 3)
         : D == 192 ? 3
                    : (cfg == 1 ? 4 : cfg == 3 ? 2 : 3);
}

struct DenseLaunch {
    DenseArgs args;
    const void *k;
    const void *v;
    int D;
    int cfg;  // mma.sync configuration 0..kDenseCfgs-1, or kUmmaCfg
    cudaStream_t stream;
    cudaEvent_t ev_before;  // measurement hook: recorded around the split kernel when both are set
    cudaEvent_t ev_after;
};

// Encodes the TMA descriptor of a [B, Skv, Hkv, D] bf16 tensor with a
// (64 x 1 x box_keys x 1) box and 128-byte swizzle.  Returns false on failure.
bool make_kv_tensor_map(CUtensorMap *map, const void *base, int B, int Skv, int Hkv, int D, int box_keys);

// Per head-dimension launchers (one translation unit each).
cudaError_t launch_dense_d64(const DenseLaunch &L);
cudaError_t launch_dense_d128(const DenseLaunch &L);
cudaError_t launch_dense_d256(const DenseLaunch &L);
// Score head size 192, value head size 128 (mma.sync engine).
cudaError_t launch_dense_d192x128(const DenseLaunch &L);
int dense_ctas_per_sm_d192x128(int cfg);
// Resident CTAs per SM of the dense split kernel for (D, cfg); 0 on error.
// cfg = kUmmaCfg gives the tcgen05 engine's figure (D = 128 and 256).
int dense_ctas_per_sm_d64(int cfg);
int dense_ctas_per_sm_d128(int cfg);
int dense_ctas_per_sm_d256(int cfg);

// Paged kernel.  Heads per CTA: the smallest power of two covering Hkv, at
// most the number whose row pieces fit 1 KiB per token (8 heads of 128 with
// 8-bit codes, 4 bf16 heads of 128), and at most 4 when a consumer holds two
// n-tiles.
// CTAs of a TMEM-allocating kernel that fit on one SM: the least of what its
// shared memory, registers, threads and TMEM columns allow.  (The CUDA
// occupancy query answers 1 for every kernel that allocates TMEM.)  The
// kernel's dynamic shared-memory limit must have been raised already.
inline int tmem_kernel_ctas_per_sm(const void *kern, int smem_bytes, int threads, int tmem_cols) {
    int dev = 0, smem_sm = 0, smem_rsv = 0, regs_sm = 0, threads_sm = 0;
    cudaFuncAttributes fa;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&smem_rsv, cudaDevAttrReservedSharedMemoryPerBlock, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&regs_sm, cudaDevAttrMaxRegistersPerMultiprocessor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&threads_sm, cudaDevAttrMaxThreadsPerMultiProcessor, dev) != cudaSuccess ||
        cudaFuncGetAttributes(&fa, kern) != cudaSuccess)
        return 0;
    const int by_smem = smem_sm / (smem_bytes + int(fa.sharedSizeBytes) + smem_rsv);
    const int regs_warp = ((fa.numRegs * 32 + 255) / 256) * 256;  // allocation unit: 256 per warp
    const int by_regs = regs_sm / (regs_warp * (threads / 32));
    const int by_threads = threads_sm / threads;
    const int by_tmem = 512 / tmem_cols;
    int n = by_smem < by_regs ? by_smem : by_regs;
    n = n < by_threads ? n : by_threads;
    return n < by_tmem ? n : by_tmem;
}
inline int paged_heads_per_cta(int D, bool kv8, int Mq, int Hkv) {
    int cap = 1024 / (D * (kv8 ? 1 : 2));
    if (cap > 8) cap = 8;
    if (Mq > 8 && cap > 4) cap = 4;
    int hb = 1;
    while (hb < Hkv && hb < cap) hb *= 2;
    return hb;
}
// The paged kernels' tcgen05 engine (gqa_paged_umma.cuh) serves FP8 pools of
// head dim 128 whose KV heads come in blocks of 8 (one 1 KiB row piece per
// token) with at most 4 query rows per KV head, in both the top-K and the
// whole-request form; other shapes run on the mma.sync engine.  (Measured on
// GB300: with 1-4 rows per KV head the tcgen05 engine is 3-16 % faster; with
// 8 rows, where two CTAs per SM leave room for only a single P buffer and
// two-stage rings, it was 4-60 % slower, so that shape stays on mma.sync.)
// Both engines use 8 heads per CTA for these shapes, so the schedule, the
// partials and the merge pass are the same.
inline bool paged_shape_fits_umma(bool fp8, int D, int Hkv, int Mq) {
    return fp8 && D == 128 && Hkv % 8 == 0 && Mq <= 4;
}
// Query rows per KV head of the instance: Mq rounded up to 2 or 4.
inline int paged_umma_rows(int Mq) { return Mq <= 2 ? 2 : 4; }
cudaError_t launch_paged_umma(const PagedArgs &a, bool range, cudaStream_t stream);
// Resident CTAs per SM (also raises the dynamic shared-memory limit on the
// current device); 0 on error.
int paged_umma_ctas_per_sm(int Mq, bool range);
cudaError_t launch_paged_topk_fp8(const PagedArgs &a, int D, cudaStream_t stream);
int paged_topk_ctas_per_sm_fp8(const PagedArgs &a, int D);
cudaError_t launch_paged_topk_combine_fp8(const PagedArgs &a, int D, cudaStream_t stream);
cudaError_t launch_paged_range_fp8(const PagedArgs &a, int D, cudaStream_t stream);
cudaError_t launch_paged_range_bf16(const PagedArgs &a, int D, cudaStream_t stream);
int paged_range_ctas_per_sm_fp8(const PagedArgs &a, int D);
int paged_range_ctas_per_sm_bf16(const PagedArgs &a, int D);
cudaError_t launch_paged_range_combine_fp8(const PagedArgs &a, int D, cudaStream_t stream);
cudaError_t launch_paged_range_int8(const PagedArgs &a, int D, cudaStream_t stream);
int paged_range_ctas_per_sm_int8(const PagedArgs &a, int D);
cudaError_t launch_paged_range_combine_int8(const PagedArgs &a, int D, cudaStream_t stream);
cudaError_t launch_paged_range_combine_bf16(const PagedArgs &a, int D, cudaStream_t stream);
cudaError_t launch_paged_gather(const uint8_t *pool, const int32_t *page_table, const int32_t *topk, uint8_t *out,
                                int B, int Hkv, int D, int page_size, int pages_per_req, int num_pages, int topk_n,
                                unsigned *err, cudaStream_t stream);
cudaError_t launch_fp8_to_f32(const uint8_t *codes, float *out, int n, cudaStream_t stream);

}  // namespace gqa
