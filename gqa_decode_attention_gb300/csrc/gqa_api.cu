// gqa_api.cu -- the C ABI front end of libgqa_decode.so.
//
// Validation, the split-count heuristic, workspace handling, TMA descriptor
// encoding and kernel dispatch.  No entry point synchronises except
// gqa_device_status and gqa_decode_host.
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "../../include/gqa_decode.h"
#include "../../include/gqa_decode_debug.h"
#include "gqa_launch.h"

namespace gqa {

__device__ unsigned g_error_word = 0;

namespace {

constexpr uint64_t kDefaultWaitLimitNs = 2000000000ull;
std::atomic<uint64_t> g_wait_limit_ns{kDefaultWaitLimitNs};
std::atomic<int> g_fault_mode{0};
std::atomic<int> g_paged_engine{0};  // 0: by shape; 1: the mma.sync engine for every paged call
std::atomic<cudaEvent_t> g_ev_before{nullptr};
std::atomic<cudaEvent_t> g_ev_after{nullptr};

constexpr int kMaxDevices = 64;
constexpr int kMinBlocksPerSplit = 2;
// Fixed cost of a wave of tcgen05 split CTAs, in 64-key blocks of walk.
// Fitted on GB300 to eight shapes (d128 Sq 8-16 and d256 Sq 8, 1-64 units,
// explicit split counts): any value from 13 to 16 picks the fastest count
// measured for each; without it the choice took 2-4 waves of short splits
// where one wave was 3-14 % faster (batch 8, 32/2 heads, d256, 128K keys:
// 333.8 -> 323.6 us; batch 8, 64/8 heads, d128 Sq 8, 8K keys: 75.8 -> 65.5 us).
#ifndef GQA_UMMA_WAVE_FIXED_BLOCKS
#define GQA_UMMA_WAVE_FIXED_BLOCKS 14
#endif
constexpr long kUmmaWaveFixedBlocks = GQA_UMMA_WAVE_FIXED_BLOCKS;
constexpr long kCtasPerSmTarget = 4;
constexpr int kMaxSplits = 4096;
constexpr long kMaxGroupRows = 4096;

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// ------------------------------------------------------------ device facts
std::mutex g_mu;
int g_sm_count[kMaxDevices];
int g_occ[kMaxDevices][4][kLaneCfg + kLaneCfgs];  // mma.sync configurations, tcgen05, key lanes

bool current_device(int *dev) {
    if (cudaGetDevice(dev) != cudaSuccess) return false;
    return *dev >= 0 && *dev < kMaxDevices;
}

int sm_count(int dev) {
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_sm_count[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        g_sm_count[dev] = n;
    }
    return g_sm_count[dev];
}

int d_index(int D) { return D == 64 ? 0 : D == 128 ? 1 : D == 192 ? 3 : 2; }

unsigned *g_err_ptr[kMaxDevices];

// Device address of the error word on `dev` (the current device).
unsigned *error_word(int dev) {
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_err_ptr[dev] == nullptr) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_error_word) != cudaSuccess) {
            cudaGetLastError();
            return nullptr;
        }
        g_err_ptr[dev] = static_cast<unsigned *>(p);
    }
    return g_err_ptr[dev];
}

// Library-owned stream-ordered memory pool per device.  It keeps freed blocks
// (release threshold = max) so the per-call workspace allocation is a cheap
// pool hit after the first call, without touching the device's default pool.
cudaMemPool_t g_pool[kMaxDevices];

cudaError_t pool_alloc(void **p, size_t bytes, int dev, cudaStream_t stream) {
    {
        std::lock_guard<std::mutex> lk(g_mu);
        if (g_pool[dev] == nullptr) {
            cudaMemPoolProps props;
            std::memset(&props, 0, sizeof(props));
            props.allocType = cudaMemAllocationTypePinned;
            props.handleTypes = cudaMemHandleTypeNone;
            props.location.type = cudaMemLocationTypeDevice;
            props.location.id = dev;
            cudaMemPool_t pool;
            cudaError_t e = cudaMemPoolCreate(&pool, &props);
            if (e != cudaSuccess) return e;
            uint64_t keep = ~uint64_t(0);
            cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &keep);
            g_pool[dev] = pool;
        }
    }
    return cudaMallocFromPoolAsync(p, bytes, g_pool[dev], stream);
}

int dense_occupancy(int dev, int D, int cfg) {
    std::lock_guard<std::mutex> lk(g_mu);
    int &slot = g_occ[dev][d_index(D)][cfg];
    if (slot == 0) {
        slot = D == 64    ? dense_ctas_per_sm_d64(cfg)
               : D == 128 ? dense_ctas_per_sm_d128(cfg)
               : D == 192 ? dense_ctas_per_sm_d192x128(cfg)
                          : dense_ctas_per_sm_d256(cfg);
    }
    return slot;
}

// ------------------------------------------------------------ TMA encoding
using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return static_cast<EncodeTiledFn>(nullptr);
        return reinterpret_cast<EncodeTiledFn>(p);
    }();
    return fn;
}

// ------------------------------------------------------------ dense shapes
struct DenseShape {
    int B, Sq, Skv, Hq, Hkv, D, G, Mq, cfg, qrows, row_groups, n_blocks;  // blocks of kSplitKeys keys
    int Dv;  // value head size (= D except for the d192x128 flavour)
};

// D: score head size (q, K); Dv: value head size (V, out).  Supported:
// D = Dv in {64, 128, 256}, and D = 192 with Dv = 128.
gqa_status check_dense_dv(int B, int Sq, int Skv, int Hq, int Hkv, int D, int Dv, DenseShape *s) {
    if (B < 1 || Sq < 1 || Skv < 1 || Hq < 1 || Hkv < 1) return GQA_ERR_INVALID_ARG;
    if (Hq % Hkv != 0 || Sq > Skv) return GQA_ERR_INVALID_ARG;
    const bool same = D == Dv && (D == 64 || D == 128 || D == 256);
    if (!same && !(D == 192 && Dv == 128)) return GQA_ERR_UNSUPPORTED;
    s->Dv = Dv;
    const long G = Hq / Hkv;
    const long Mq = G * Sq;
    if (Mq > kMaxGroupRows) return GQA_ERR_UNSUPPORTED;
    if (long(Skv) * Hkv >= (1L << 31)) return GQA_ERR_UNSUPPORTED;
    if (B > 65535) return GQA_ERR_UNSUPPORTED;
    s->B = B;
    s->Sq = Sq;
    s->Skv = Skv;
    s->Hq = Hq;
    s->Hkv = Hkv;
    s->D = D;
    s->G = int(G);
    s->Mq = int(Mq);
    s->cfg = dense_uses_umma(D, Dv, Sq) ? kUmmaCfg : dense_cfg_for_rows(int(Mq < 128 ? Mq : 128));
    s->qrows = dense_rows_per_cta(s->cfg);
    s->row_groups = int((Mq + s->qrows - 1) / s->qrows);
    if (long(Hkv) * s->row_groups > 65535) return GQA_ERR_UNSUPPORTED;
    s->n_blocks = (Skv + kSplitKeys - 1) / kSplitKeys;
    return GQA_OK;
}

gqa_status check_dense(int B, int Sq, int Skv, int Hq, int Hkv, int D, DenseShape *s) {
    return check_dense_dv(B, Sq, Skv, Hq, Hkv, D, D, s);
}

// Split count.  The kernel is HBM-bound once about kCtasPerSmTarget CTAs are
// resident on every SM (enough loads in flight), so:
//  - units (batch x KV head x row group) already giving that many CTAs: 1
//    split; with small CTAs (kCtasPerSmTarget or more resident) already at
//    three quarters of that many (measured on GB300 at 512 units against 608:
//    1 split 3-6 % faster than 2, which leave a partial second wave);
//  - otherwise the fewest splits that reach the target while the whole grid
//    stays one wave of resident CTAs;
//  - when occupancy is too low for that (large CTAs), the split count that
//    minimises waves x key blocks per CTA, i.e. balanced waves.
// Every split covers at least kMinBlocksPerSplit blocks of 64 keys, at most
// kMaxSplits splits are used, and the count is then evened out so that all
// splits but the last cover the same number of blocks.
int choose_splits(const DenseShape &s, int requested, int dev) {
    int S;
    if (requested > 0) {
        S = requested;
    } else {
        const long units = long(s.B) * s.Hkv * s.row_groups;
        const long nsm = sm_count(dev) > 0 ? sm_count(dev) : 1;
        const long occ = dense_occupancy(dev, s.D, s.cfg) > 0 ? dense_occupancy(dev, s.D, s.cfg) : 1;
        const long slots = nsm * occ;
        const long target = nsm * (occ < kCtasPerSmTarget ? occ : kCtasPerSmTarget);
        const long max_s = (s.n_blocks + kMinBlocksPerSplit - 1) / kMinBlocksPerSplit;
        if (units >= target || (occ >= kCtasPerSmTarget && 4 * units >= 3 * target)) {
            S = 1;
        } else {
            const long s_min = (target + units - 1) / units;
            const long s_one_wave = slots / units;
            if (s_min <= s_one_wave) {
                S = int(s_min);
            } else {
                // a wave of tcgen05 CTAs also pays a fixed start and finish
                // (TMEM, queries, the first tiles, the epilogue)
                const long fixed = s.cfg == kUmmaCfg ? kUmmaWaveFixedBlocks : 0;
                long best = 1, best_cost = -1;
                for (long c = 1; c <= 4 * s_one_wave + 4 && c <= max_s; ++c) {
                    const long waves = (units * c + slots - 1) / slots;
                    const long cost = waves * ((s.n_blocks + c - 1) / c + fixed);
                    if (best_cost < 0 || cost < best_cost) {
                        best_cost = cost;
                        best = c;
                    }
                }
                S = int(best);
            }
        }
        if (S > max_s) S = int(max_s);
    }
    if (S > s.n_blocks) S = s.n_blocks;
    if (S > kMaxSplits) S = kMaxSplits;
    return S < 1 ? 1 : S;
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

size_t workspace_bytes(const DenseShape &s, int splits) {
    if (splits <= 1) return 0;
    const size_t rows = size_t(s.B) * s.Hkv * splits * s.Mq;
    return align256(rows * s.Dv * sizeof(float)) + align256(rows * sizeof(float));
}

// key blocks per split as the kernel sees it for a split count
int blocks_per_split(const DenseShape &s, int splits) { return (s.n_blocks + splits - 1) / splits; }

// What one call launches: the split count (as realised by blocks_per_split),
// key blocks per split, and the kernel configuration.  An explicit split count
// is always honoured as given.  Otherwise, where the automatic choice would
// split the cache and the units (batch row, KV head, row group) are few, the
// key-lane instance takes over: its CTA fills an SM and its warps split the
// walk, so
//  - a cache of at most GQA_LANE_MAX_UNIT_BYTES per unit runs as one CTA per
//    unit (one launch, no combine pass), as long as the units fit one wave;
//  - a longer cache is split across one wave of key-lane CTAs (SMs / units
//    splits, combined when there are several) when the units are at most a
//    quarter of the SMs; when that wave fills at least 80 % of the SMs with
//    one CTA per unit (no combine pass), or with several whose splits hold at
//    least GQA_LANE_MIN_SPLIT_KEYS keys; or when one CTA per unit fills 60 %
//    of the SMs with caches of at most that many keys.
// Measured on GB300 (device time per call, L2 flushed): batch 1 with 8 KV
// heads and 1K-8K keys went from 16-18 us to 14 us, and the 128K-key
// two-row decode from 92 to 87 us; with 64-72 units (batch 8-9, two splits a
// unit) splits of 2K keys and more were 2-7 % faster than the general choice
// and shorter ones up to 1 us slower, and a wave of 120 CTAs (batch 5, three
// splits) was 2 us slower at 8K-16K keys; with 128-152 units (batch 16-19,
// one key-lane CTA a unit) 600-32K keys were 4-26 % faster; with 96-112 units
// (63-74 % of the SMs) 1K-2K keys were 4-14 % faster and 4K keys and more
// 7-50 % slower (one SM then pulls a whole unit).
struct DensePlan {
    int splits, tps, cfg;
};
#ifndef GQA_LANE_MIN_SPLITS
#define GQA_LANE_MIN_SPLITS 4
#endif
#ifndef GQA_LANE_ONE_WAVE
#define GQA_LANE_ONE_WAVE 1  // 0: small caches only (tuning builds)
#endif
#ifndef GQA_LANE_MIN_SPLIT_KEYS
#define GQA_LANE_MIN_SPLIT_KEYS 2048
#endif

DensePlan plan_dense(const DenseShape &s, int requested, int dev) {
    const int splits = choose_splits(s, requested, dev);
    const long units = long(s.B) * s.Hkv * s.row_groups;
    const long nsm = sm_count(dev) > 0 ? sm_count(dev) : 1;
    const bool lanes_fit = requested == 0 && splits > 1 && dense_has_lanes(s.D, s.Dv) &&
                           s.cfg < dense_lane_row_cfgs(s.D, s.Dv) && units <= nsm;
    if (lanes_fit && long(s.Skv) * (s.D + s.Dv) * 2 <= long(GQA_LANE_MAX_UNIT_BYTES))
        return {1, s.n_blocks, dense_lane_cfg_for(s.cfg, true)};
    const long per_sm = nsm / units;  // key-lane splits a unit gets in one wave
    const long fill_pct = 100 * units * per_sm / nsm;  // SMs the wave occupies
    const bool one_wave_lanes = GQA_LANE_ONE_WAVE && (
        per_sm >= GQA_LANE_MIN_SPLITS ||
        (fill_pct >= 80 && (per_sm == 1 || long(s.Skv) / per_sm >= GQA_LANE_MIN_SPLIT_KEYS)) ||
        (per_sm == 1 && fill_pct >= 60 && s.Skv <= GQA_LANE_MIN_SPLIT_KEYS));
    if (lanes_fit && one_wave_lanes) {
        long ls = per_sm;
        if (ls > kMaxSplits) ls = kMaxSplits;
        if (ls > s.n_blocks) ls = s.n_blocks;
        const int ltps = blocks_per_split(s, int(ls));
        return {(s.n_blocks + ltps - 1) / ltps, ltps, dense_lane_cfg_for(s.cfg, false)};
    }
    const int tps = blocks_per_split(s, splits);
    return {(s.n_blocks + tps - 1) / tps, tps, s.cfg};
}

gqa_status run_dense(const void *q, const void *k, const void *v, void *out, float *lse, const DenseShape &s,
                     float scale, int requested_splits, void *workspace, size_t workspace_size,
                     cudaStream_t stream) {
    int dev = 0;
    if (!current_device(&dev)) return GQA_ERR_CUDA;
    if (encode_fn() == nullptr) return GQA_ERR_CUDA;
    // The first occupancy query on a device also raises the kernel's dynamic
    // shared-memory limit there (a per-device attribute); made here so that a
    // call with an explicit split count on a second device is covered too.
    dense_occupancy(dev, s.D, s.cfg);
    const DensePlan plan = plan_dense(s, requested_splits, dev);
    if (plan.cfg != s.cfg) dense_occupancy(dev, s.D, plan.cfg);  // raises that kernel's limit too
    const int splits = plan.splits;
    const int tps = plan.tps;
    const size_t need = workspace_bytes(s, splits);
    void *ws = workspace;
    bool owned = false;
    if (need > 0) {
        if (ws != nullptr) {
            if (workspace_size < need) return GQA_ERR_NO_MEMORY;
            if (!aligned(ws, 256)) return GQA_ERR_ALIGNMENT;
        } else {
            if (pool_alloc(&ws, need, dev, stream) != cudaSuccess) {
                cudaGetLastError();
                return GQA_ERR_NO_MEMORY;
            }
            owned = true;
        }
    }
    DenseLaunch L;
    std::memset(&L, 0, sizeof(L));
    DenseArgs &a = L.args;
    a.q = static_cast<const __nv_bfloat16 *>(q);
    a.out = static_cast<__nv_bfloat16 *>(out);
    a.lse = lse;
    if (need > 0) {
        const size_t rows = size_t(s.B) * s.Hkv * splits * s.Mq;
        a.o_part = static_cast<float *>(ws);
        a.lse_part = reinterpret_cast<float *>(static_cast<char *>(ws) + align256(rows * s.Dv * sizeof(float)));
    }
    a.B = s.B;
    a.Sq = s.Sq;
    a.Skv = s.Skv;
    a.Hq = s.Hq;
    a.Hkv = s.Hkv;
    a.G = s.G;
    a.Mq = s.Mq;
    a.n_blocks = s.n_blocks;
    a.blocks_per_split = tps;
    a.num_splits = splits;
    a.row_groups = s.row_groups;
    a.alpha = scale * 1.4426950408889634f;
    a.wait_limit_ns = g_wait_limit_ns.load();
    a.fault_mode = g_fault_mode.load();
    a.err = error_word(dev);
    L.k = k;
    L.v = v;
    L.D = s.D;
    L.cfg = plan.cfg;
    L.stream = stream;
    L.ev_before = g_ev_before.load();
    L.ev_after = g_ev_after.load();
    cudaError_t e = s.D == 64    ? launch_dense_d64(L)
                    : s.D == 128 ? launch_dense_d128(L)
                    : s.D == 192 ? launch_dense_d192x128(L)
                                 : launch_dense_d256(L);
    if (owned) cudaFreeAsync(ws, stream);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return GQA_ERR_CUDA;
    }
    return GQA_OK;
}

float resolve_scale(float scale, int D) {
    if (!(scale > 0.f) || std::isinf(scale)) return 1.0f / std::sqrt(float(D));
    return scale;
}

gqa_status check_dense_ptrs(const void *q, const void *k, const void *v, const void *out, const float *lse) {
    if (q == nullptr || k == nullptr || v == nullptr || out == nullptr) return GQA_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16) || !aligned(lse, 4))
        return GQA_ERR_ALIGNMENT;
    return GQA_OK;
}

// ------------------------------------------------------------ paged checks
gqa_status check_paged(int B, int Hq, int Hkv, int D, int page_size, int pages_per_req, int num_pages, int topk) {
    if (B < 1 || Hq < 1 || Hkv < 1 || page_size < 1 || pages_per_req < 1 || num_pages < 1 || topk < 0)
        return GQA_ERR_INVALID_ARG;
    if (Hq % Hkv != 0) return GQA_ERR_INVALID_ARG;
    if (long(topk) > long(pages_per_req) * page_size) return GQA_ERR_INVALID_ARG;
    if (D != 64 && D != 128 && D != 256) return GQA_ERR_UNSUPPORTED;
    if (long(pages_per_req) * page_size >= (1L << 31)) return GQA_ERR_UNSUPPORTED;
    if (long(num_pages) * page_size >= (1L << 31)) return GQA_ERR_UNSUPPORTED;
    if (topk > 65536 || B > 65535) return GQA_ERR_UNSUPPORTED;
    return GQA_OK;
}

// ------------------------------------------------------------ paged, whole requests

struct PagedShape {
    int B, Sq, Hq, Hkv, D, G, Mq, ps, ppr, num_pages, cap;
    int kvt;         // GQA_KV_BF16 / GQA_KV_FP8_E4M3FN / GQA_KV_INT8
    bool kv8;        // 8-bit codes (FP8 or int8)
    bool topk_form;  // the sparse top-K form (FP8, gated) rather than whole requests
};

// The paged engine a shape runs on: tcgen05 where the shape fits it (unless
// the measurement hook asks for the mma.sync engine everywhere).
bool paged_umma(const PagedShape &s) {
    return g_paged_engine.load() == 0 && paged_shape_fits_umma(s.kvt == GQA_KV_FP8_E4M3FN, s.D, s.Hkv, s.Mq);
}

gqa_status check_paged_kv(int B, int Sq, int Hq, int Hkv, int D, int kv_dtype, int page_size, int pages_per_req,
                          int num_pages, PagedShape *s) {
    if (B < 1 || Sq < 1 || Hq < 1 || Hkv < 1 || page_size < 1 || pages_per_req < 1 || num_pages < 1)
        return GQA_ERR_INVALID_ARG;
    if (Hq % Hkv != 0) return GQA_ERR_INVALID_ARG;
    if (kv_dtype != GQA_KV_BF16 && kv_dtype != GQA_KV_FP8_E4M3FN && kv_dtype != GQA_KV_INT8)
        return GQA_ERR_INVALID_ARG;
    if (D != 64 && D != 128) return GQA_ERR_UNSUPPORTED;
    const long G = Hq / Hkv;
    if (G * Sq > 16) return GQA_ERR_UNSUPPORTED;
    if (long(pages_per_req) * page_size >= (1L << 31) || long(num_pages) * page_size >= (1L << 31))
        return GQA_ERR_UNSUPPORTED;
    if (B > 65535) return GQA_ERR_UNSUPPORTED;
    s->B = B;
    s->Sq = Sq;
    s->Hq = Hq;
    s->Hkv = Hkv;
    s->D = D;
    s->G = int(G);
    s->Mq = int(G * Sq);
    s->ps = page_size;
    s->ppr = pages_per_req;
    s->num_pages = num_pages;
    s->cap = pages_per_req * page_size;
    s->kvt = kv_dtype;
    s->kv8 = kv_dtype != GQA_KV_BF16;
    s->topk_form = false;
    return GQA_OK;
}

// Resident CTAs per SM of the paged instance serving shape s (cached).
int paged_occupancy(int dev, const PagedShape &s) {
    static int cache[kMaxDevices][4][2][2][4];  // [dev][form][D][two n-tiles][log2 heads per CTA]
    static int cache_umma[kMaxDevices][2][2];   // tcgen05 engine: [dev][whole-request form][rows 2 / 4]
    const int hb = paged_heads_per_cta(s.D, s.kv8, s.Mq, s.Hkv);
    const int lh = hb == 1 ? 0 : hb == 2 ? 1 : hb == 4 ? 2 : 3;
    const int form = s.topk_form ? 3 : s.kvt;
    std::lock_guard<std::mutex> lk(g_mu);
    if (paged_umma(s)) {
        const int R = paged_umma_rows(s.Mq);
        int &u = cache_umma[dev][s.topk_form ? 0 : 1][R == 2 ? 0 : 1];
        if (u == 0) u = paged_umma_ctas_per_sm(s.Mq, !s.topk_form);
        return u;
    }
    int &slot = cache[dev][form][s.D == 128][s.Mq > 8][lh];
    if (slot == 0) {
        PagedArgs a;
        std::memset(&a, 0, sizeof(a));
        a.Hkv = s.Hkv;
        a.Mq = s.Mq;
        slot = s.topk_form                  ? paged_topk_ctas_per_sm_fp8(a, s.D)
               : s.kvt == GQA_KV_INT8        ? paged_range_ctas_per_sm_int8(a, s.D)
               : s.kvt == GQA_KV_FP8_E4M3FN ? paged_range_ctas_per_sm_fp8(a, s.D)
                                            : paged_range_ctas_per_sm_bf16(a, s.D);
    }
    return slot;
}

// Workers per head block of the balanced schedule: one resident CTA slot
// each (the kernel is bound by bytes in flight, so every slot should stream),
// at least one.  The top-K form (equal lists) uses one worker per request as
// soon as the requests fill half the slots: a request then never straddles
// two workers and no merge pass is needed, which costs less than the idle
// slots it leaves (measured on both engines).
int choose_paged_workers(const PagedShape &s, int requested, int dev) {
    long W;
    if (requested > 0) {
        W = requested;
    } else {
        const int hb = paged_heads_per_cta(s.D, s.kv8, s.Mq, s.Hkv);
        const long nhb = (s.Hkv + hb - 1) / hb;
        const long nsm = sm_count(dev) > 0 ? sm_count(dev) : 1;
        const long occ = paged_occupancy(dev, s) > 0 ? paged_occupancy(dev, s) : 1;
        W = nsm * occ / nhb;
#ifndef GQA_PAGED_TOPK_ONE_PER_REQUEST
#define GQA_PAGED_TOPK_ONE_PER_REQUEST 1
#endif
        if (GQA_PAGED_TOPK_ONE_PER_REQUEST && s.topk_form && 2 * long(s.B) * nhb >= nsm * occ) W = s.B;
    }
    if (W > 65535) W = 65535;
    return W < 1 ? 1 : int(W);
}

// Partials of the shared requests: per (head block, worker) two slots (the
// worker's first and last segment) of HB heads x Mq rows.
size_t paged_workspace_bytes(const PagedShape &s, int workers) {
    if (workers <= 1) return 0;
    const int hb = paged_heads_per_cta(s.D, s.kv8, s.Mq, s.Hkv);
    const size_t nhb = (s.Hkv + hb - 1) / hb;
    const size_t rows = nhb * size_t(workers) * 2 * hb * s.Mq;
    const size_t prefix = s.topk_form ? 0 : align256((size_t(s.B) + 1) * sizeof(long long));
    return align256(rows * s.D * sizeof(float)) + align256(rows * sizeof(float)) + prefix;
}

// Points the kernel arguments at the partial buffers inside a workspace of
// paged_workspace_bytes(s, workers) bytes.
void paged_bind_workspace(const PagedShape &s, int workers, void *ws, PagedArgs *a) {
    const int hb = paged_heads_per_cta(s.D, s.kv8, s.Mq, s.Hkv);
    const size_t rows = size_t((s.Hkv + hb - 1) / hb) * workers * 2 * hb * s.Mq;
    char *p = static_cast<char *>(ws);
    a->o_part = reinterpret_cast<float *>(p);
    p += align256(rows * s.D * sizeof(float));
    a->lse_part = reinterpret_cast<float *>(p);
    p += align256(rows * sizeof(float));
    a->step_prefix = s.topk_form ? nullptr : reinterpret_cast<long long *>(p);
}

}  // namespace

// K or V as a 4-D tensor (d, kv head, key, batch) with a box of 64 head-dim
// elements (128 bytes, one swizzle atom) x 1 head x box_keys keys x 1 batch.
// Keys past Skv read as zeros.
bool make_kv_tensor_map(CUtensorMap *map, const void *base, int B, int Skv, int Hkv, int D, int box_keys) {
    EncodeTiledFn enc = encode_fn();
    if (enc == nullptr) return false;
    const cuuint64_t dims[4] = {cuuint64_t(D), cuuint64_t(Hkv), cuuint64_t(Skv), cuuint64_t(B)};
    const cuuint64_t strides[3] = {cuuint64_t(D) * 2, cuuint64_t(Hkv) * D * 2, cuuint64_t(Skv) * Hkv * D * 2};
    const cuuint32_t box[4] = {64, 1, cuuint32_t(box_keys), 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(base), dims, strides, box,
                           estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

}  // namespace gqa

using namespace gqa;

extern "C" {

const char *gqa_status_string(gqa_status s) {
    switch (s) {
        case GQA_OK: return "GQA_OK";
        case GQA_ERR_INVALID_ARG: return "GQA_ERR_INVALID_ARG";
        case GQA_ERR_UNSUPPORTED: return "GQA_ERR_UNSUPPORTED";
        case GQA_ERR_ALIGNMENT: return "GQA_ERR_ALIGNMENT";
        case GQA_ERR_NO_MEMORY: return "GQA_ERR_NO_MEMORY";
        case GQA_ERR_CUDA: return "GQA_ERR_CUDA";
        case GQA_ERR_DEVICE_TIMEOUT: return "GQA_ERR_DEVICE_TIMEOUT";
        case GQA_ERR_DEVICE_INDEX: return "GQA_ERR_DEVICE_INDEX";
    }
    return "GQA_ERR_UNKNOWN";
}

const char *gqa_version(void) { return "gqa_decode 0.1.0 (sm_103a)"; }

gqa_status gqa_decode_ex(const void *q, const void *k, const void *v, void *out, float *lse, int B, int Sq, int Skv,
                         int Hq, int Hkv, int D, float scale, int num_splits, void *workspace,
                         size_t workspace_bytes_, gqa_stream_t stream) {
    DenseShape s;
    gqa_status st = check_dense(B, Sq, Skv, Hq, Hkv, D, &s);
    if (st != GQA_OK) return st;
    if (num_splits < 0) return GQA_ERR_INVALID_ARG;
    st = check_dense_ptrs(q, k, v, out, lse);
    if (st != GQA_OK) return st;
    return run_dense(q, k, v, out, lse, s, resolve_scale(scale, D), num_splits, workspace, workspace_bytes_,
                     reinterpret_cast<cudaStream_t>(stream));
}

gqa_status gqa_decode_dv(const void *q, const void *k, const void *v, void *out, float *lse, int B, int Sq, int Skv,
                         int Hq, int Hkv, int Dqk, int Dv, float scale, int num_splits, void *workspace,
                         size_t workspace_bytes_, gqa_stream_t stream) {
    DenseShape s;
    gqa_status st = check_dense_dv(B, Sq, Skv, Hq, Hkv, Dqk, Dv, &s);
    if (st != GQA_OK) return st;
    if (num_splits < 0) return GQA_ERR_INVALID_ARG;
    st = check_dense_ptrs(q, k, v, out, lse);
    if (st != GQA_OK) return st;
    return run_dense(q, k, v, out, lse, s, resolve_scale(scale, Dqk), num_splits, workspace, workspace_bytes_,
                     reinterpret_cast<cudaStream_t>(stream));
}

size_t gqa_decode_dv_workspace_bytes(int B, int Sq, int Skv, int Hq, int Hkv, int Dqk, int Dv, int num_splits) {
    DenseShape s;
    if (check_dense_dv(B, Sq, Skv, Hq, Hkv, Dqk, Dv, &s) != GQA_OK || num_splits < 0) return 0;
    int dev = 0;
    if (num_splits == 0 && !current_device(&dev)) return 0;
    return workspace_bytes(s, plan_dense(s, num_splits, dev).splits);
}

gqa_status gqa_decode(const void *q, const void *k, const void *v, void *out, float *lse, int B, int Sq, int Skv,
                      int Hq, int Hkv, int D, float scale, gqa_stream_t stream) {
    return gqa_decode_ex(q, k, v, out, lse, B, Sq, Skv, Hq, Hkv, D, scale, 0, nullptr, 0, stream);
}

int gqa_decode_num_splits(int B, int Sq, int Skv, int Hq, int Hkv, int D) {
    return gqa_decode_dv_num_splits(B, Sq, Skv, Hq, Hkv, D, D);
}

int gqa_decode_dv_num_splits(int B, int Sq, int Skv, int Hq, int Hkv, int Dqk, int Dv) {
    DenseShape s;
    gqa_status st = check_dense_dv(B, Sq, Skv, Hq, Hkv, Dqk, Dv, &s);
    if (st != GQA_OK) return -int(st);
    int dev = 0;
    if (!current_device(&dev)) return -int(GQA_ERR_CUDA);
    return plan_dense(s, 0, dev).splits;
}

int gqa_decode_dense_engine(int B, int Sq, int Skv, int Hq, int Hkv, int Dqk, int Dv) {
    DenseShape s;
    gqa_status st = check_dense_dv(B, Sq, Skv, Hq, Hkv, Dqk, Dv, &s);
    if (st != GQA_OK) return -int(st);
    return s.cfg == kUmmaCfg ? GQA_ENGINE_TCGEN05 : GQA_ENGINE_MMA_SYNC;
}

size_t gqa_decode_workspace_bytes(int B, int Sq, int Skv, int Hq, int Hkv, int D, int num_splits) {
    DenseShape s;
    if (check_dense(B, Sq, Skv, Hq, Hkv, D, &s) != GQA_OK || num_splits < 0) return 0;
    int dev = 0;
    if (num_splits == 0 && !current_device(&dev)) return 0;
    return workspace_bytes(s, plan_dense(s, num_splits, dev).splits);
}

gqa_status gqa_decode_host(const void *q_host, const void *k_host, const void *v_host, void *out_host,
                           float *lse_host, int B, int Sq, int Skv, int Hq, int Hkv, int D, float scale,
                           gqa_stream_t stream_) {
    DenseShape s;
    gqa_status st = check_dense(B, Sq, Skv, Hq, Hkv, D, &s);
    if (st != GQA_OK) return st;
    if (q_host == nullptr || k_host == nullptr || v_host == nullptr || out_host == nullptr)
        return GQA_ERR_INVALID_ARG;
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    const size_t qb = size_t(B) * Sq * Hq * D * 2;
    const size_t kvb = size_t(B) * Skv * Hkv * D * 2;
    const size_t lb = size_t(B) * Hq * Sq * sizeof(float);
    const size_t total = align256(qb) + 2 * align256(kvb) + align256(qb) + align256(lb);
    char *base = nullptr;
    int dev = 0;
    if (!current_device(&dev)) return GQA_ERR_CUDA;
    if (pool_alloc(reinterpret_cast<void **>(&base), total, dev, stream) != cudaSuccess) {
        cudaGetLastError();
        return GQA_ERR_NO_MEMORY;
    }
    char *dq = base;
    char *dk = dq + align256(qb);
    char *dv = dk + align256(kvb);
    char *dout = dv + align256(kvb);
    float *dlse = reinterpret_cast<float *>(dout + align256(qb));
    gqa_status result = GQA_OK;
    if (cudaMemcpyAsync(dq, q_host, qb, cudaMemcpyHostToDevice, stream) != cudaSuccess ||
        cudaMemcpyAsync(dk, k_host, kvb, cudaMemcpyHostToDevice, stream) != cudaSuccess ||
        cudaMemcpyAsync(dv, v_host, kvb, cudaMemcpyHostToDevice, stream) != cudaSuccess) {
        result = GQA_ERR_CUDA;
    }
    if (result == GQA_OK)
        result = run_dense(dq, dk, dv, dout, lse_host ? dlse : nullptr, s, resolve_scale(scale, D), 0, nullptr, 0,
                           stream);
    if (result == GQA_OK) {
        if (cudaMemcpyAsync(out_host, dout, qb, cudaMemcpyDeviceToHost, stream) != cudaSuccess ||
            (lse_host && cudaMemcpyAsync(lse_host, dlse, lb, cudaMemcpyDeviceToHost, stream) != cudaSuccess))
            result = GQA_ERR_CUDA;
    }
    cudaFreeAsync(base, stream);
    if (cudaStreamSynchronize(stream) != cudaSuccess && result == GQA_OK) result = GQA_ERR_CUDA;
    if (result == GQA_ERR_CUDA) cudaGetLastError();
    return result;
}

}  // extern "C"

namespace {

// The sparse top-K form: host scalars k_scale / v_scale, or (k_scales,
// v_scales, n_scales) in device memory (n_scales 1 or Hkv), which multiply
// the host scalars.
gqa_status run_paged_topk(const void *q, const void *gate, const uint8_t *k_pool, const uint8_t *v_pool,
                          const int32_t *page_table, const int32_t *topk_idx, float k_scale, float v_scale,
                          const float *k_scales, const float *v_scales, int n_scales, void *out, float *lse, int B,
                          int Hq, int Hkv, int D, int page_size, int pages_per_req, int num_pages, int topk,
                          float scale, gqa_stream_t stream) {
    gqa_status st = check_paged(B, Hq, Hkv, D, page_size, pages_per_req, num_pages, topk);
    if (st != GQA_OK) return st;
    if (D == 256 || Hq / Hkv > 16) return GQA_ERR_UNSUPPORTED;
    if (!std::isfinite(k_scale) || !std::isfinite(v_scale)) return GQA_ERR_INVALID_ARG;
    if (k_scales != nullptr || v_scales != nullptr) {
        if (k_scales == nullptr || v_scales == nullptr || (n_scales != 1 && n_scales != Hkv))
            return GQA_ERR_INVALID_ARG;
        if (!aligned(k_scales, 4) || !aligned(v_scales, 4)) return GQA_ERR_ALIGNMENT;
    }
    if (q == nullptr || gate == nullptr || k_pool == nullptr || v_pool == nullptr || out == nullptr ||
        page_table == nullptr || (topk > 0 && topk_idx == nullptr))
        return GQA_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(gate, 16) || !aligned(k_pool, 16) || !aligned(v_pool, 16) ||
        !aligned(out, 16) || !aligned(lse, 4) || !aligned(page_table, 4) || !aligned(topk_idx, 4))
        return GQA_ERR_ALIGNMENT;
    PagedArgs a;
    std::memset(&a, 0, sizeof(a));
    a.q = static_cast<const __nv_bfloat16 *>(q);
    a.gate = static_cast<const __nv_bfloat16 *>(gate);
    a.k_pool = k_pool;
    a.v_pool = v_pool;
    a.page_table = page_table;
    a.topk = topk_idx;
    a.out = static_cast<__nv_bfloat16 *>(out);
    a.lse = lse;
    a.B = B;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.G = Hq / Hkv;
    a.page_size = page_size;
    a.pages_per_req = pages_per_req;
    a.num_pages = num_pages;
    a.topk_n = topk;
    a.Sq = 1;
    a.Mq = a.G;
    a.alpha = resolve_scale(scale, D) * k_scale * 1.4426950408889634f;
    a.v_scale = v_scale;
    a.k_scales = k_scales;
    a.v_scales = v_scales;
    a.n_scales = k_scales != nullptr ? n_scales : 0;
    a.wait_limit_ns = g_wait_limit_ns.load();
    a.fault_mode = g_fault_mode.load();
    int dev = 0;
    if (!current_device(&dev)) return GQA_ERR_CUDA;
    a.err = error_word(dev);
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    // Balanced schedule: one worker per resident CTA slot per head block.
    PagedShape ps_;
    std::memset(&ps_, 0, sizeof(ps_));
    ps_.B = B;
    ps_.Sq = 1;
    ps_.Hq = Hq;
    ps_.Hkv = Hkv;
    ps_.D = D;
    ps_.G = a.G;
    ps_.Mq = a.G;
    ps_.kvt = GQA_KV_FP8_E4M3FN;
    ps_.kv8 = true;
    ps_.topk_form = true;
    const int workers = choose_paged_workers(ps_, 0, dev);
    a.num_splits = workers;
    // Equal lists: a request is shared by two workers only when some worker
    // boundary floor(w T / W) falls inside it.
    bool shared = false;
    {
        const long steps = (long(topk) + kPagedStageTokens - 1) / kPagedStageTokens;
        const long T = steps * B;
        for (long w = 1; w < workers && steps > 0 && !shared; ++w) shared = (w * T / workers) % steps != 0;
    }
    const size_t need = shared ? paged_workspace_bytes(ps_, workers) : 0;
    void *ws = nullptr;
    if (need > 0) {
        if (pool_alloc(&ws, need, dev, cs) != cudaSuccess) {
            cudaGetLastError();
            return GQA_ERR_NO_MEMORY;
        }
        paged_bind_workspace(ps_, workers, ws, &a);
    }
    cudaEvent_t eb = g_ev_before.load(), ea = g_ev_after.load();
    if (eb != nullptr && ea != nullptr) cudaEventRecord(eb, cs);
    cudaError_t pe = paged_umma(ps_) ? launch_paged_umma(a, false, cs) : launch_paged_topk_fp8(a, D, cs);
    if (eb != nullptr && ea != nullptr) cudaEventRecord(ea, cs);
    if (pe == cudaSuccess && shared) pe = launch_paged_topk_combine_fp8(a, D, cs);
    if (ws != nullptr) cudaFreeAsync(ws, cs);
    if (pe != cudaSuccess) {
        cudaGetLastError();
        return GQA_ERR_CUDA;
    }
    return GQA_OK;
}

}  // namespace

extern "C" {

gqa_status gqa_decode_paged_fp8(const void *q, const void *gate, const uint8_t *k_pool, const uint8_t *v_pool,
                                const int32_t *page_table, const int32_t *topk_idx, float k_scale, float v_scale,
                                void *out, float *lse, int B, int Hq, int Hkv, int D, int page_size,
                                int pages_per_req, int num_pages, int topk, float scale, gqa_stream_t stream) {
    return run_paged_topk(q, gate, k_pool, v_pool, page_table, topk_idx, k_scale, v_scale, nullptr, nullptr, 0, out,
                          lse, B, Hq, Hkv, D, page_size, pages_per_req, num_pages, topk, scale, stream);
}

gqa_status gqa_decode_paged_fp8_dev_scales(const void *q, const void *gate, const uint8_t *k_pool,
                                           const uint8_t *v_pool, const int32_t *page_table,
                                           const int32_t *topk_idx, const float *k_scales, const float *v_scales,
                                           int n_scales, void *out, float *lse, int B, int Hq, int Hkv, int D,
                                           int page_size, int pages_per_req, int num_pages, int topk, float scale,
                                           gqa_stream_t stream) {
    if (k_scales == nullptr || v_scales == nullptr) return GQA_ERR_INVALID_ARG;
    return run_paged_topk(q, gate, k_pool, v_pool, page_table, topk_idx, 1.0f, 1.0f, k_scales, v_scales, n_scales,
                          out, lse, B, Hq, Hkv, D, page_size, pages_per_req, num_pages, topk, scale, stream);
}

namespace {
gqa_status run_paged_kv(const void *q, const void *k_pool, const void *v_pool, int kv_dtype, float k_scale,
                        float v_scale, const float *k_scales, const float *v_scales, int n_scales,
                        const int32_t *page_table, const int32_t *seq_lens, void *out, float *lse, int B, int Sq,
                        int Hq, int Hkv, int D, int page_size, int pages_per_req, int num_pages, float scale,
                        int num_splits, void *workspace, size_t workspace_bytes_, gqa_stream_t stream) {
    PagedShape s;
    gqa_status st = check_paged_kv(B, Sq, Hq, Hkv, D, kv_dtype, page_size, pages_per_req, num_pages, &s);
    if (st != GQA_OK) return st;
    if (num_splits < 0) return GQA_ERR_INVALID_ARG;
    if (s.kv8 && (!std::isfinite(k_scale) || !std::isfinite(v_scale))) return GQA_ERR_INVALID_ARG;
    if (k_scales != nullptr || v_scales != nullptr) {
        if (k_scales == nullptr || v_scales == nullptr || (n_scales != 1 && n_scales != Hkv))
            return GQA_ERR_INVALID_ARG;
        if (!aligned(k_scales, 4) || !aligned(v_scales, 4)) return GQA_ERR_ALIGNMENT;
    }
    if (q == nullptr || k_pool == nullptr || v_pool == nullptr || page_table == nullptr || seq_lens == nullptr ||
        out == nullptr)
        return GQA_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(k_pool, 16) || !aligned(v_pool, 16) || !aligned(out, 16) || !aligned(lse, 4) ||
        !aligned(page_table, 4) || !aligned(seq_lens, 4))
        return GQA_ERR_ALIGNMENT;
    int dev = 0;
    if (!current_device(&dev)) return GQA_ERR_CUDA;
    paged_occupancy(dev, s);  // sets the kernel's shared-memory limit on this device (see run_dense)
    const int splits = choose_paged_workers(s, num_splits, dev);
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    const size_t need = paged_workspace_bytes(s, splits);
    void *ws = workspace;
    bool owned = false;
    if (need > 0) {
        if (ws != nullptr) {
            if (workspace_bytes_ < need) return GQA_ERR_NO_MEMORY;
            if (!aligned(ws, 256)) return GQA_ERR_ALIGNMENT;
        } else {
            if (pool_alloc(&ws, need, dev, cs) != cudaSuccess) {
                cudaGetLastError();
                return GQA_ERR_NO_MEMORY;
            }
            owned = true;
        }
    }
    PagedArgs a;
    std::memset(&a, 0, sizeof(a));
    a.q = static_cast<const __nv_bfloat16 *>(q);
    a.k_pool = static_cast<const uint8_t *>(k_pool);
    a.v_pool = static_cast<const uint8_t *>(v_pool);
    a.page_table = page_table;
    a.seq_lens = seq_lens;
    a.out = static_cast<__nv_bfloat16 *>(out);
    a.lse = lse;
    if (need > 0) paged_bind_workspace(s, splits, ws, &a);
    a.B = B;
    a.Sq = Sq;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.G = s.G;
    a.Mq = s.Mq;
    a.page_size = page_size;
    a.pages_per_req = pages_per_req;
    a.num_pages = num_pages;
    a.num_splits = splits;
    a.alpha = resolve_scale(scale, D) * (s.kv8 ? k_scale : 1.0f) * 1.4426950408889634f;
    a.v_scale = s.kv8 ? v_scale : 1.0f;
    a.k_scales = k_scales;
    a.v_scales = v_scales;
    a.n_scales = n_scales;
    a.wait_limit_ns = g_wait_limit_ns.load();
    a.fault_mode = g_fault_mode.load();
    a.err = error_word(dev);
    cudaEvent_t eb = g_ev_before.load(), ea = g_ev_after.load();
    if (eb != nullptr && ea != nullptr) cudaEventRecord(eb, cs);
    cudaError_t e = paged_umma(s)                ? launch_paged_umma(a, true, cs)
                    : s.kvt == GQA_KV_INT8        ? launch_paged_range_int8(a, D, cs)
                    : s.kvt == GQA_KV_FP8_E4M3FN ? launch_paged_range_fp8(a, D, cs)
                                                 : launch_paged_range_bf16(a, D, cs);
    if (eb != nullptr && ea != nullptr) cudaEventRecord(ea, cs);
    if (e == cudaSuccess && splits > 1)
        e = s.kvt == GQA_KV_INT8        ? launch_paged_range_combine_int8(a, D, cs)
            : s.kvt == GQA_KV_FP8_E4M3FN ? launch_paged_range_combine_fp8(a, D, cs)
                                         : launch_paged_range_combine_bf16(a, D, cs);
    if (owned) cudaFreeAsync(ws, cs);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return GQA_ERR_CUDA;
    }
    return GQA_OK;
}
}  // namespace

gqa_status gqa_decode_paged_ex(const void *q, const void *k_pool, const void *v_pool, int kv_dtype, float k_scale,
                               float v_scale, const int32_t *page_table, const int32_t *seq_lens, void *out,
                               float *lse, int B, int Sq, int Hq, int Hkv, int D, int page_size, int pages_per_req,
                               int num_pages, float scale, int num_splits, void *workspace,
                               size_t workspace_bytes_, gqa_stream_t stream) {
    return run_paged_kv(q, k_pool, v_pool, kv_dtype, k_scale, v_scale, nullptr, nullptr, 0, page_table, seq_lens,
                        out, lse, B, Sq, Hq, Hkv, D, page_size, pages_per_req, num_pages, scale, num_splits,
                        workspace, workspace_bytes_, stream);
}

gqa_status gqa_decode_paged_dev_scales(const void *q, const void *k_pool, const void *v_pool, int kv_dtype,
                                       const float *k_scales, const float *v_scales, int n_scales,
                                       const int32_t *page_table, const int32_t *seq_lens, void *out, float *lse,
                                       int B, int Sq, int Hq, int Hkv, int D, int page_size, int pages_per_req,
                                       int num_pages, float scale, int num_splits, void *workspace,
                                       size_t workspace_bytes_, gqa_stream_t stream) {
    if (kv_dtype == GQA_KV_BF16 || k_scales == nullptr || v_scales == nullptr) return GQA_ERR_INVALID_ARG;
    return run_paged_kv(q, k_pool, v_pool, kv_dtype, 1.0f, 1.0f, k_scales, v_scales, n_scales, page_table,
                        seq_lens, out, lse, B, Sq, Hq, Hkv, D, page_size, pages_per_req, num_pages, scale,
                        num_splits, workspace, workspace_bytes_, stream);
}

gqa_status gqa_decode_paged(const void *q, const void *k_pool, const void *v_pool, int kv_dtype, float k_scale,
                            float v_scale, const int32_t *page_table, const int32_t *seq_lens, void *out, float *lse,
                            int B, int Sq, int Hq, int Hkv, int D, int page_size, int pages_per_req, int num_pages,
                            float scale, gqa_stream_t stream) {
    return gqa_decode_paged_ex(q, k_pool, v_pool, kv_dtype, k_scale, v_scale, page_table, seq_lens, out, lse, B, Sq,
                               Hq, Hkv, D, page_size, pages_per_req, num_pages, scale, 0, nullptr, 0, stream);
}

int gqa_decode_paged_num_splits(int B, int Sq, int Hq, int Hkv, int D, int kv_dtype, int page_size,
                                int pages_per_req) {
    PagedShape s;
    gqa_status st = check_paged_kv(B, Sq, Hq, Hkv, D, kv_dtype, page_size, pages_per_req, 1, &s);
    if (st != GQA_OK) return -int(st);
    int dev = 0;
    if (!current_device(&dev)) return -int(GQA_ERR_CUDA);
    return choose_paged_workers(s, 0, dev);
}

size_t gqa_decode_paged_workspace_bytes(int B, int Sq, int Hq, int Hkv, int D, int kv_dtype, int page_size,
                                        int pages_per_req, int num_splits) {
    PagedShape s;
    if (check_paged_kv(B, Sq, Hq, Hkv, D, kv_dtype, page_size, pages_per_req, 1, &s) != GQA_OK || num_splits < 0)
        return 0;
    int dev = 0;
    if (num_splits == 0 && !current_device(&dev)) return 0;
    return paged_workspace_bytes(s, choose_paged_workers(s, num_splits, dev));
}

gqa_status gqa_paged_gather_fp8(const uint8_t *pool, const int32_t *page_table, const int32_t *topk_idx, uint8_t *out,
                                int B, int Hkv, int D, int page_size, int pages_per_req, int num_pages, int topk,
                                gqa_stream_t stream) {
    gqa_status st = check_paged(B, Hkv, Hkv, D, page_size, pages_per_req, num_pages, topk);
    if (st != GQA_OK) return st;
    if (pool == nullptr || page_table == nullptr || out == nullptr || (topk > 0 && topk_idx == nullptr))
        return GQA_ERR_INVALID_ARG;
    if (!aligned(pool, 16) || !aligned(out, 16) || !aligned(page_table, 4) || !aligned(topk_idx, 4))
        return GQA_ERR_ALIGNMENT;
    if (topk == 0) return GQA_OK;
    int dev = 0;
    if (!current_device(&dev)) return GQA_ERR_CUDA;
    if (launch_paged_gather(pool, page_table, topk_idx, out, B, Hkv, D, page_size, pages_per_req, num_pages, topk,
                            error_word(dev), reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) {
        cudaGetLastError();
        return GQA_ERR_CUDA;
    }
    return GQA_OK;
}

gqa_status gqa_fp8_e4m3fn_to_f32(const uint8_t *codes, float *out, int n, gqa_stream_t stream) {
    if (n < 0 || (n > 0 && (codes == nullptr || out == nullptr))) return GQA_ERR_INVALID_ARG;
    if (!aligned(out, 4)) return GQA_ERR_ALIGNMENT;
    if (n == 0) return GQA_OK;
    if (launch_fp8_to_f32(codes, out, n, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) {
        cudaGetLastError();
        return GQA_ERR_CUDA;
    }
    return GQA_OK;
}

gqa_status gqa_device_status(gqa_stream_t stream) {
    if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) {
        cudaGetLastError();
        return GQA_ERR_CUDA;
    }
    unsigned word = 0;
    const unsigned zero = 0;
    if (cudaMemcpyFromSymbol(&word, g_error_word, sizeof(word)) != cudaSuccess ||
        cudaMemcpyToSymbol(g_error_word, &zero, sizeof(zero)) != cudaSuccess) {
        cudaGetLastError();
        return GQA_ERR_CUDA;
    }
    if (word & kErrTimeout) return GQA_ERR_DEVICE_TIMEOUT;
    if (word & kErrIndex) return GQA_ERR_DEVICE_INDEX;
    return GQA_OK;
}

void gqa_set_wait_limit_ns(uint64_t ns) {
    constexpr uint64_t kMinWaitLimitNs = 1000000ull;
    g_wait_limit_ns.store(ns == 0 ? kDefaultWaitLimitNs : ns < kMinWaitLimitNs ? kMinWaitLimitNs : ns);
}

void gqa_debug_set_fault_mode(int mode) { g_fault_mode.store(mode); }

int gqa_decode_paged_engine(int B, int Sq, int Hq, int Hkv, int D, int kv_dtype, int topk_form) {
    PagedShape s;
    std::memset(&s, 0, sizeof(s));
    if (topk_form) {
        gqa_status st = check_paged(B, Hq, Hkv, D, 1, 1, 1, 0);
        if (st != GQA_OK) return -int(st);
        if (D == 256 || Hq / Hkv > 16) return -int(GQA_ERR_UNSUPPORTED);
        s.B = B;
        s.Sq = 1;
        s.Hq = Hq;
        s.Hkv = Hkv;
        s.D = D;
        s.G = Hq / Hkv;
        s.Mq = s.G;
        s.kvt = GQA_KV_FP8_E4M3FN;
        s.kv8 = true;
        s.topk_form = true;
    } else {
        gqa_status st = check_paged_kv(B, Sq, Hq, Hkv, D, kv_dtype, 1, 1, 1, &s);
        if (st != GQA_OK) return -int(st);
    }
    return paged_umma(s) ? GQA_ENGINE_TCGEN05 : GQA_ENGINE_MMA_SYNC;
}

void gqa_debug_set_paged_engine(int mode) { g_paged_engine.store(mode == 1 ? 1 : 0); }

void gqa_debug_set_kernel_events(void *before, void *after) {
    g_ev_before.store(static_cast<cudaEvent_t>(before));
    g_ev_after.store(static_cast<cudaEvent_t>(after));
}

}  // extern "C"
