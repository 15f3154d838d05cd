// gqa_paged_umma.cuh -- paged GQA decode over an FP8 E4M3FN pool on the
// fifth-generation tensor cores (tcgen05 + TMEM): the sparse top-K form with a
// sigmoid output gate ("Sparse paged GQA decode attention with FP8 KV cache
// on SM89", sections "Workload" and "Implementations") and the whole-request
// form, for pools of 8 (or a multiple of 8) KV heads of 128 dimensions and at
// most 4 query rows per KV head.
//
// What it computes is what gqa_paged_kernel computes (same schedule, same
// partials, same merge pass); only the data path differs.
//
// Data path.  A CTA serves a block of 8 KV heads.  Its producer warps gather
// the selected tokens with one bulk asynchronous copy per token of the
// token's whole 1 KiB K row piece (8 heads x 128 codes) and one of its V
// piece, 16 tokens per ring stage: the copy engine moves whole contiguous
// rows, the fastest of the gathers measured on this machine (per-head 128-byte
// tile gathers and 16-byte copies ran 5-15 % slower).  The tensor core reads
// those rows as they landed:
//   scores  S^T[(t, g) x (g', r)] = K_raw[(t, g) x 128] . Q'[(g', r) x 128]^T
//           M = 128 = 16 tokens x 8 heads (one TMEM lane per token and head),
//           N = 8 heads x R query rows, K = 128 codes; entries with g' = g
//           are the scores, the rest are discarded;
//   output  O^T[d x (g, r)] += V_raw^T[d x (t, g')] . P'^T[(t, g') x (g, r)]
//           with P' block-diagonal (zero unless g' = g), so one product sums
//           every head's weighted values into its own columns.
// Both operands are described to the tensor core as 128-byte-swizzled tiles,
// which they are not: the hardware then reads 16-byte chunk c of row m from
// position c ^ (m mod 8), and since m mod 8 is the head g of the row, every
// head's dimensions arrive permuted by "xor g" at 16-byte granularity.  A dot
// product is unchanged when both sides are permuted alike, so Q' holds each
// head's query rows permuted the same way; in the output product the
// permutation moves head g's output dimensions, which the epilogue maps back.
//
// Precision.  The MMA kind is f8f6f4 (E4M3 x E4M3, fp32 accumulation), so K
// and V codes enter the tensor core as they are stored.  The 16-bit query
// row, scaled by a power of two so its largest element lies in [128, 256),
// is split into two E4M3 values q = hi + lo (exact to bf16's precision for
// every element within 2^-9 of the row maximum); both products accumulate
// into the same scores.  The weights p = 2^6 exp2(x - m) (m the running
// reference maximum, rescaled lazily) are split as hi = e4m3(p) and
// lo = e4m3(16 (p - hi)) into two output accumulators, O = O_hi + O_lo / 16:
// relative error about 2^-8 per weight, and weights below about 2^-20 of the
// row's reference maximum are dropped.  The normaliser sums the unrounded
// fp32 weights.
//
// Roles (8 warps):
//   warps 0-3   softmax: thread = TMEM lane m = 8 t + g (token t of the 16,
//               head g of the 8); the epilogue stages O through shared
//               memory and writes whole 16-byte pieces of output rows.
//   warp 4      allocates TMEM; lane 0 issues every MMA as its inputs become
//               ready, the output product of the oldest block first, then the
//               next score product (two S buffers in TMEM).
//   warp 5      copies K and warp 6 copies V into separate rings: one bulk
//               copy per token row piece, or one per block when its 16 rows
//               are consecutive pool rows.
//   warp 7      index map: the pool rows and token masks of the coming blocks,
//               four blocks per round (two memory latencies a round).
// Every wait is bounded in wall time; on expiry the CTA flags the device
// error word, stops, drains its own copies and MMAs, frees TMEM and returns.
#pragma once

#include "gqa_common.cuh"
#include "gqa_paged_kernel.cuh"
#include "gqa_params.h"
#include "gqa_umma.cuh"

namespace gqa {

// Instruction descriptor of tcgen05.mma kind::f8f6f4 with E4M3 A and B and
// fp32 D; a_mn / b_mn select the MN-major layout of A / B.
__host__ __device__ constexpr uint32_t idesc_e4m3_f32(int M, int N, bool a_mn, bool b_mn) {
    return (1u << 4)                        // D format: f32
           | (0u << 7) | (0u << 10)         // A, B format: E4M3
           | (uint32_t(a_mn) << 15) | (uint32_t(b_mn) << 16)
           | (uint32_t(N >> 3) << 17) | (uint32_t(M >> 4) << 24);
}

// Shared-memory matrix descriptor without swizzling (layout type 0).  For an
// MN-major operand the core matrices are 8 rows (K) x 16 bytes (MN): lbo is
// the byte distance between core matrices along K, sbo along MN.
__device__ __forceinline__ uint64_t smem_desc_plain(uint32_t addr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = 0;
    d |= uint64_t((addr & 0x3FFFFu) >> 4);
    d |= uint64_t((lbo >> 4) & 0x3FFFu) << 16;
    d |= uint64_t((sbo >> 4) & 0x3FFFu) << 32;
    d |= uint64_t(1) << 46;
    return d;
}

// D[tmem] (+)= A[smem] * B[smem], kind::f8f6f4; issued by one thread.
__device__ __forceinline__ void umma_e4m3(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                          uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Two floats to two E4M3 codes (lo -> low byte), round to nearest even,
// saturating at +-448.
__device__ __forceinline__ uint16_t f32x2_to_e4m3x2(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

// The two E4M3 values of a pair of codes, as floats (exact).
__device__ __forceinline__ float2 e4m3x2_to_f32x2(uint16_t two) {
    const uint32_t h = e4m3x2_to_f16x2(two);
    return __half22float2(*reinterpret_cast<const __half2 *>(&h));
}

// Named barrier of the 128 softmax threads; `bar.red.or` returns whether the
// predicate held on any of them.
__device__ __forceinline__ void softmax_bar() { asm volatile("bar.sync 1, 128;" ::: "memory"); }
__device__ __forceinline__ bool softmax_bar_any(bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, 1, 128, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(uint32_t(pred))
        : "memory");
    return r != 0;
}

template <int R>
struct PagedUmmaCfg {
    static_assert(R == 2 || R == 4 || R == 8, "query rows per KV head: 2, 4 or 8 (8 is not instantiated)");
    static constexpr int HB = 8;                  // KV heads per CTA
    static constexpr int D = 128;                 // head dim (one 128-byte FP8 row per head)
    static constexpr int BT = kPagedStageTokens;  // tokens per block: M = 128 = BT x HB
    static_assert(BT * HB == 128, "one TMEM lane per token and head");
    static constexpr int N = HB * R;              // score / output columns
    static constexpr int PIECE = HB * D;          // bytes of a token's row piece (K or V)
    static constexpr int KV_BYTES = BT * PIECE;   // K (or V) of one block
    // Separate K and V rings: a K stage is free once its scores are computed,
    // a V stage only after the block's softmax and output product, so the K
    // ring runs further ahead.  Depths fill two CTAs' shared memory per SM.
#ifndef GQA_PAGED_UMMA_KST4
#define GQA_PAGED_UMMA_KST4 2
#endif
#ifndef GQA_PAGED_UMMA_VST4
#define GQA_PAGED_UMMA_VST4 3
#endif
    static constexpr int KST = R == 2 ? 3 : R == 4 ? GQA_PAGED_UMMA_KST4 : 2;
    static constexpr int VST = R == 2 ? 3 : R == 4 ? GQA_PAGED_UMMA_VST4 : 2;
    static constexpr int Q_BYTES = N * 128;       // one E4M3 piece of Q' (N rows of 128 codes)
    static constexpr int P_BYTES = 128 * N;       // one E4M3 piece of P'^T (128 rows x N bytes)
    static constexpr int P_BUFS = R <= 4 ? 2 : 1;
    static constexpr int OUT_PIECES = N * D / 8;   // 16-byte pieces of the output rows (bf16)
    static_assert(N * D * 4 <= P_BUFS * 2 * P_BYTES, "the epilogue stages O (fp32) over the P buffers");
    static_assert(OUT_PIECES % 128 == 0, "whole rounds of output pieces");
    static constexpr int P_NBLK = 2048;           // P'^T: byte distance between 16-column blocks
    static constexpr float kPExp = 6.f;           // p = 2^kPExp exp2(x - m)
    static constexpr float kLazy = 2.75f;         // rescale once x exceeds m by more than this
    static constexpr int NP = 3;                  // producer warps: K, V, index map
    static constexpr int IDX_SLOTS = 8;           // blocks of pool rows the index warp resolves ahead
    // Token masks of the blocks, written by the index warp, read by the softmax.
    // The index warp writes block j only after both copy warps read block
    // j - IDX_SLOTS, and the V warp gets there only after the output product
    // of block j - IDX_SLOTS - 1 - VST, i.e. after the softmax finished it: the
    // index warp runs at most IDX_SLOTS + VST + 1 blocks ahead of the softmax,
    // fewer than VM_SLOTS.
    static constexpr int VM_SLOTS = 16;
    static constexpr int SW = 0;                  // first softmax warp (lane quarter = warp)
    static constexpr int ISSUER = 4;
    static constexpr int PW0 = 5;                 // first producer warp
    static constexpr int THREADS = 32 * (PW0 + NP);
    // shared memory (from a 1024-byte aligned base)
    static constexpr int K_OFF = 0;
    static constexpr int V_OFF = K_OFF + KST * KV_BYTES;
    static constexpr int Q_OFF = V_OFF + VST * KV_BYTES;
    static constexpr int P_OFF = Q_OFF + 2 * Q_BYTES;
    static constexpr int BAR_OFF = P_OFF + P_BUFS * 2 * P_BYTES;
    // barriers: kfull[KST], kempty[KST], vfull[VST], vempty[VST], s_full[2], s_free[2],
    // p_full[PB], pv_done[PB], q_full, o_free, fin, idx_full[IDX_SLOTS], idx_empty[IDX_SLOTS],
    // vm_full[VM_SLOTS]
    static constexpr int NBARS = 2 * KST + 2 * VST + 4 + 2 * P_BUFS + 3 + 2 * IDX_SLOTS + VM_SLOTS;
    static constexpr int VMASK_OFF = BAR_OFF + NBARS * 8;           // u32 per block slot (valid tokens)
    static constexpr int ALPHA_OFF = VMASK_OFF + VM_SLOTS * 4;      // float [N]
    static constexpr int MREF_OFF = ALPHA_OFF + N * 4;              // float [N] reference maxima
    static constexpr int CORR_OFF = MREF_OFF + N * 4;               // float [N]
    static constexpr int XCH_OFF = CORR_OFF + N * 4;                // float [2][4][N] block maxima
    static constexpr int LSUM_OFF = XCH_OFF + 2 * 4 * N * 4;        // float [4][N]
    static constexpr int SCHED_OFF = (LSUM_OFF + 4 * N * 4 + 7) / 8 * 8;  // long [4]
    static constexpr int MISC_OFF = SCHED_OFF + 32;                 // tmem base, abort flag
    static constexpr int IDX_OFF = MISC_OFF + 16;                   // int [IDX_SLOTS][BT] pool rows
    static constexpr int COLB_OFF = (IDX_OFF + IDX_SLOTS * BT * 4 + 7) / 8 * 8;  // long long [N] output row offsets
    static constexpr int COLF_OFF = COLB_OFF + N * 8;               // float [N] output factors
    static constexpr int SMEM_USED = COLF_OFF + N * 4;
    static constexpr int SMEM_BYTES = SMEM_USED + 1024;             // + alignment slack
    // TMEM columns: two score buffers, then O_hi and O_lo
    static constexpr uint32_t S_COL = 0;
    static constexpr uint32_t OH_COL = 2 * N;
    static constexpr uint32_t OL_COL = 3 * N;
    static constexpr uint32_t TMEM_COLS = 4 * N <= 64 ? 64 : 4 * N <= 128 ? 128 : 256;
    static constexpr int MIN_BLOCKS = (2 * (SMEM_BYTES + 1024) <= 228 * 1024) ? 2 : 1;
};

// ---------------------------------------------------------------- schedule
// The balanced schedule of the paged kernels, computed once per CTA: worker
// w = blockIdx.y of W = num_splits takes the global 16-token steps
// [w T / W, (w + 1) T / W) of all requests (T of them), in request order.
// Returns (through the arguments) its step range and its first request and
// that request's first global step; the whole-request form also records, in
// worker 0 of head block 0, every request's first step for the merge pass.
template <bool RANGE>
__device__ __forceinline__ void paged_schedule(const PagedArgs &a, long *sched, int warp, int lane, long &w_begin,
                                               long &w_end, int &seg_b, long &seg_p) {
    if constexpr (!RANGE) {
        const long steps = (a.topk_n + kPagedStageTokens - 1) / kPagedStageTokens;
        const long T = steps * a.B;
        const int W = a.num_splits;
        w_begin = long(blockIdx.y) * T / W;
        w_end = (long(blockIdx.y) + 1) * T / W;
        seg_b = steps > 0 ? int(w_begin / steps) : 0;
        seg_p = long(seg_b) * steps;
    } else {
        if (warp == 0) {
            const int W = a.num_splits;
            const int cap = a.pages_per_req * a.page_size;
            long T = 0;
            for (int b0 = 0; b0 < a.B; b0 += 32) {
                const int bb = b0 + lane;
                int len = bb >= a.B ? 0 : __ldg(a.seq_lens + bb);
                len = len < 0 ? 0 : (len > cap ? cap : len);
                long st = (len + kPagedStageTokens - 1) / kPagedStageTokens;
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) st += __shfl_xor_sync(0xffffffffu, st, off);
                T += st;
            }
            if (a.step_prefix != nullptr && blockIdx.x == 0 && blockIdx.y == 0) {
                long Q = 0;
                for (int b0 = 0; b0 < a.B; b0 += 32) {
                    const int bb = b0 + lane;
                    int len = bb < a.B ? __ldg(a.seq_lens + bb) : 0;
                    len = len < 0 ? 0 : (len > cap ? cap : len);
                    const long st = (len + kPagedStageTokens - 1) / kPagedStageTokens;
                    long incl = st;
#pragma unroll
                    for (int off = 1; off < 32; off <<= 1) {
                        const long y = __shfl_up_sync(0xffffffffu, incl, off);
                        if (lane >= off) incl += y;
                    }
                    if (bb < a.B) a.step_prefix[bb] = Q + incl - st;
                    Q += __shfl_sync(0xffffffffu, incl, 31);
                }
                if (lane == 0) a.step_prefix[a.B] = Q;
            }
            const long start = long(blockIdx.y) * T / W, end = (long(blockIdx.y) + 1) * T / W;
            long P = 0;
            int first = a.B;
            long first_p = T;
            for (int b0 = 0; b0 < a.B && first == a.B; b0 += 32) {
                const int bb = b0 + lane;
                int len = bb >= a.B ? 0 : __ldg(a.seq_lens + bb);
                len = len < 0 ? 0 : (len > cap ? cap : len);
                const long st = (len + kPagedStageTokens - 1) / kPagedStageTokens;
                long incl = st;
#pragma unroll
                for (int off = 1; off < 32; off <<= 1) {
                    const long y = __shfl_up_sync(0xffffffffu, incl, off);
                    if (lane >= off) incl += y;
                }
                // an empty request at step P counts as reaching P + 1: the worker
                // whose range holds P writes it (the last worker when P = T)
                const bool hit = bb < a.B && P + incl - st + (st > 0 ? st : 1) > start;
                const unsigned m = __ballot_sync(0xffffffffu, hit);
                if (m != 0u) {
                    const int l = __ffs(m) - 1;
                    first = b0 + l;
                    first_p = P + __shfl_sync(0xffffffffu, incl - st, l);
                }
                P += __shfl_sync(0xffffffffu, incl, 31);
            }
            if (lane == 0) {
                sched[0] = start;
                sched[1] = end;
                sched[2] = first;
                sched[3] = first_p;
            }
        }
        __syncthreads();
        w_begin = sched[0];
        w_end = sched[1];
        seg_b = int(sched[2]);
        seg_p = sched[3];
    }
}

// Walks the segments of a worker's step range: segment = (request b, its
// tokens [t_begin, t_begin + n_tok)), complete when it is the whole request,
// slot 0 for the worker's first segment and 1 otherwise.  Every role of the
// CTA walks the same sequence.
struct PagedSegWalk {
    long w_begin, w_end, seg_t, seg_p;
    int seg_b;
    bool last_worker;
    // current segment (valid after next() returned true)
    int b, seq_len, t_begin, n_tok, nblk, slot;
    bool complete;
    long seg_next, steps_b;
    bool bad;

    __device__ __forceinline__ void init(long wb, long we, int sb, long sp, bool last) {
        w_begin = wb;
        w_end = we;
        seg_t = wb;
        seg_b = sb;
        seg_p = sp;
        last_worker = last;
        bad = false;
    }
    template <bool RANGE>
    __device__ __forceinline__ bool next(const PagedArgs &a) {
        if (!(seg_b < a.B && (seg_t < w_end || (last_worker && seg_t == w_end)))) return false;
        b = seg_b;
        seq_len = RANGE ? __ldg(a.seq_lens + b) : a.topk_n;
        const int cap = a.pages_per_req * a.page_size;
        if (seq_len < 0 || seq_len > cap) {
            bad = true;
            seq_len = seq_len < 0 ? 0 : cap;
        }
        steps_b = (seq_len + kPagedStageTokens - 1) / kPagedStageTokens;
        seg_next = min(w_end, seg_p + steps_b);
        t_begin = int(seg_t - seg_p) * kPagedStageTokens;
        n_tok = min(int(seg_next - seg_p) * kPagedStageTokens, seq_len) - t_begin;
        if (n_tok < 0) n_tok = 0;
        nblk = (n_tok + kPagedStageTokens - 1) / kPagedStageTokens;
        complete = seg_t == seg_p && seg_next == seg_p + steps_b;
        slot = seg_t == w_begin ? 0 : 1;
        return true;
    }
    __device__ __forceinline__ void advance() {
        if (seg_next == seg_p + steps_b) {
            seg_p = seg_next;
            ++seg_b;
        }
        seg_t = seg_next;
    }
};

// Block-by-block walk of the same sequence: the non-empty segments' 16-token
// blocks in order; `blk` is the block within its segment and `ns` the index
// of its segment among the non-empty ones.
struct PagedBlockWalk {
    PagedSegWalk w;
    int blk, ns;
    bool in_seg;
    __device__ __forceinline__ void init(long wb, long we, int sb, long sp, bool last) {
        w.init(wb, we, sb, sp, last);
        in_seg = false;
        blk = 0;
        ns = -1;
    }
    template <bool RANGE>
    __device__ __forceinline__ bool next(const PagedArgs &a) {
        if (in_seg && blk + 1 < w.nblk) {
            ++blk;
            return true;
        }
        if (in_seg) w.advance();
        while (w.next<RANGE>(a)) {
            if (w.nblk > 0) {
                in_seg = true;
                blk = 0;
                ++ns;
                return true;
            }
            w.advance();
        }
        in_seg = false;
        return false;
    }
};

template <int R, bool RANGE>
__global__ void __launch_bounds__(PagedUmmaCfg<R>::THREADS, PagedUmmaCfg<R>::MIN_BLOCKS)
    gqa_paged_umma_kernel(const PagedArgs a) {
    using C = PagedUmmaCfg<R>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *kfull = reinterpret_cast<uint64_t *>(smem + C::BAR_OFF);
    uint64_t *kempty = kfull + C::KST;
    uint64_t *vfull = kempty + C::KST;
    uint64_t *vempty = vfull + C::VST;
    uint64_t *s_full = vempty + C::VST;    // [2]
    uint64_t *s_free = s_full + 2;         // [2]
    uint64_t *p_full = s_free + 2;         // [P_BUFS]
    uint64_t *pv_done = p_full + C::P_BUFS;  // [P_BUFS]
    uint64_t *q_full = pv_done + C::P_BUFS;
    uint64_t *o_free = q_full + 1;
    uint64_t *fin = o_free + 1;
    uint64_t *idx_full = fin + 1;              // [IDX_SLOTS]
    uint64_t *idx_empty = idx_full + C::IDX_SLOTS;
    uint64_t *vm_full = idx_empty + C::IDX_SLOTS;  // [VM_SLOTS]
    int *idx_rows = reinterpret_cast<int *>(smem + C::IDX_OFF);
    long long *col_base = reinterpret_cast<long long *>(smem + C::COLB_OFF);
    float *col_f = reinterpret_cast<float *>(smem + C::COLF_OFF);
    uint32_t *vmask = reinterpret_cast<uint32_t *>(smem + C::VMASK_OFF);
    float *alpha_s = reinterpret_cast<float *>(smem + C::ALPHA_OFF);
    float *mref_s = reinterpret_cast<float *>(smem + C::MREF_OFF);
    float *corr_s = reinterpret_cast<float *>(smem + C::CORR_OFF);
    float *xch = reinterpret_cast<float *>(smem + C::XCH_OFF);
    float *lsum = reinterpret_cast<float *>(smem + C::LSUM_OFF);
    long *sched = reinterpret_cast<long *>(smem + C::SCHED_OFF);
    uint32_t *tmem_base_s = reinterpret_cast<uint32_t *>(smem + C::MISC_OFF);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::MISC_OFF + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int hb = blockIdx.x;
    const int hb0 = hb * C::HB;  // first KV head of the block

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::KST; ++s) {
            mbar_init(&kfull[s], 1);
            mbar_init(&kempty[s], 1);  // the scores' commit
        }
        for (int s = 0; s < C::VST; ++s) {
            mbar_init(&vfull[s], 1);
            mbar_init(&vempty[s], 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(&s_full[s], 1);
            mbar_init(&s_free[s], 4);  // one arrival per softmax warp
        }
        for (int s = 0; s < C::P_BUFS; ++s) {
            mbar_init(&p_full[s], 4);
            mbar_init(&pv_done[s], 1);
        }
        mbar_init(q_full, 1);
        mbar_init(o_free, 4);
        mbar_init(fin, 1);
        for (int s = 0; s < C::IDX_SLOTS; ++s) {
            mbar_init(&idx_full[s], 1);
            mbar_init(&idx_empty[s], 2);  // the K and the V producer
        }
        for (int s = 0; s < C::VM_SLOTS; ++s) mbar_init(&vm_full[s], 1);
        *abort_flag = 0;
        fence_mbarrier_init();
    }
    // P'^T is block-diagonal: only each token-and-head row's own head columns
    // are ever written, the rest stay zero.
    for (int i = threadIdx.x; i < C::P_BUFS * 2 * C::P_BYTES / 16; i += C::THREADS)
        reinterpret_cast<uint4 *>(smem + C::P_OFF)[i] = make_uint4(0u, 0u, 0u, 0u);
    fence_proxy_async_shared();
    if (warp == C::ISSUER) tmem_alloc(tmem_base_s, C::TMEM_COLS);
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tbase = *tmem_base_s;
    pdl_wait_primary();  // inputs may be written by the previous kernel in the stream

    long w_begin, w_end, seg_p;
    int seg_b;
    paged_schedule<RANGE>(a, sched, warp, lane, w_begin, w_end, seg_b, seg_p);
    const bool last_worker = int(blockIdx.y) == a.num_splits - 1;
    const size_t row_bytes = size_t(a.Hkv) * C::D;

    if (warp == C::PW0 + 2) {
        // ============================================================ index map
        // Pool rows of the coming blocks into a ring of IDX_SLOTS blocks, four
        // blocks per round: every lane loads its two tokens' list entries (top-K
        // form) and page-table entries together, so a round costs two memory
        // latencies whatever its size, and the copy warps never wait on them.
        PagedSegWalk w;
        w.init(w_begin, w_end, seg_b, seg_p, last_worker);
        bool failed = false;
        int j = 0;
        while (!failed && w.next<RANGE>(a)) {
            for (int b0 = 0; b0 < w.nblk && !failed; b0 += 4) {
                const int nb = min(4, w.nblk - b0);
                int tk[2];
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int k = b0 * C::BT + lane + 32 * e;  // token of the segment
                    const bool in = k < (b0 + nb) * C::BT && k < w.n_tok;
                    if constexpr (RANGE)
                        tk[e] = in ? w.t_begin + k : -1;
                    else
                        tk[e] = in ? __ldg(a.topk + size_t(w.b) * a.topk_n + w.t_begin + k) : -1;
                }
                int rw[2];
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    bool bad = false;
                    rw[e] = paged_token_row(a.page_table, w.b, a.pages_per_req, a.page_size, a.num_pages, tk[e], &bad);
                    if (bad) w.bad = true;
                }
                for (int q = 0; q < nb; ++q) {
                    const int jj = j + q;
                    if (jj < C::IDX_SLOTS) continue;
                    bool ok = true;
                    if (lane == 0)
                        ok = mbar_wait_bounded(&idx_empty[jj % C::IDX_SLOTS], ((jj / C::IDX_SLOTS) - 1) & 1,
                                               a.wait_limit_ns, abort_flag);
                    if (!__shfl_sync(0xffffffffu, ok, 0)) {
                        failed = true;
                        break;
                    }
                }
                if (failed) break;
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int q = (lane >> 4) + 2 * e;  // block of the round holding this token
                    if (q < nb) idx_rows[((j + q) % C::IDX_SLOTS) * C::BT + (lane & 15)] = rw[e];
                }
                // token masks: bit i of block q = token i has a row
                const unsigned b0m = __ballot_sync(0xffffffffu, rw[0] >= 0);  // blocks 0, 1 of the round
                const unsigned b1m = __ballot_sync(0xffffffffu, rw[1] >= 0);  // blocks 2, 3
                if (lane < nb) {
                    const unsigned wm = lane < 2 ? b0m : b1m;
                    vmask[(j + lane) % C::VM_SLOTS] = (lane & 1) ? (wm >> 16) : (wm & 0xffffu);
                }
                __syncwarp();
                if (lane == 0)
                    for (int q = 0; q < nb; ++q) {
                        mbar_arrive(&idx_full[(j + q) % C::IDX_SLOTS]);
                        mbar_arrive(&vm_full[(j + q) % C::VM_SLOTS]);
                    }
                j += nb;
            }
            w.advance();
        }
        if (failed) {
            if (lane == 0) flag_error(a.err, kErrTimeout);
            *abort_flag = 1;
        }
        if (w.bad && lane == 0) flag_error(a.err, kErrIndex);
        return;
    }

    if (warp >= C::PW0) {
        // ============================================================ copy warps
        // Warp PW0 copies K, warp PW0 + 1 copies V, each into its own ring:
        // lane i < 16 one copy of token i's row piece, or lane 0 one copy of
        // the whole block when its 16 rows are consecutive pool rows of full
        // pieces (a page-aligned block of a whole request, page size a
        // multiple of 16, 8 KV heads).
        const bool is_v = warp == C::PW0 + 1;
        const int nst = is_v ? C::VST : C::KST;
        uint64_t *fullb = is_v ? vfull : kfull;
        uint64_t *emptyb = is_v ? vempty : kempty;
        const uint32_t base = smem_u32(smem + (is_v ? C::V_OFF : C::K_OFF));
        const uint8_t *pool = (is_v ? a.v_pool : a.k_pool) + size_t(hb0) * C::D;
        const bool copier = lane < C::BT;
        const bool whole_rows = a.Hkv == C::HB;  // a token's piece is its whole pool row
        PagedSegWalk w;
        w.init(w_begin, w_end, seg_b, seg_p, last_worker);
        bool failed = false;
        int jb = 0;      // global block index of this CTA
        int issued = 0;  // blocks issued so far
        while (!failed && w.next<RANGE>(a)) {
            for (int blk = 0; blk < w.nblk; ++blk, ++jb) {
                // this block's rows from the index warp
                const int slot = jb % C::IDX_SLOTS;
                bool ok = true;
                if (lane == 0) ok = mbar_wait_bounded(&idx_full[slot], (jb / C::IDX_SLOTS) & 1, a.wait_limit_ns, abort_flag);
                if (!__shfl_sync(0xffffffffu, ok, 0)) {
                    failed = true;
                    break;
                }
                const int row = copier ? idx_rows[slot * C::BT + lane] : -1;
                __syncwarp();
                if (lane == 0) mbar_arrive(&idx_empty[slot]);
                const int st = jb % nst;
                if (jb >= nst) {
                    if (lane == 0) ok = mbar_wait_bounded(&emptyb[st], ((jb / nst) - 1) & 1, a.wait_limit_ns, abort_flag);
                    if (!__shfl_sync(0xffffffffu, ok, 0)) {
                        failed = true;
                        break;
                    }
                }
                const unsigned valid = __ballot_sync(0xffffffffu, row >= 0);  // lanes 0-15
                const int r0 = __shfl_sync(0xffffffffu, row, 0);
                const bool contig =
                    whole_rows && __ballot_sync(0xffffffffu, copier && row >= 0 && row == r0 + lane) == 0xffffu;
                issued = jb + 1;
                const uint32_t dst = base + uint32_t(st * C::KV_BYTES);
                if (lane == 0) mbar_arrive_expect_tx(&fullb[st], uint32_t(__popc(valid)) * C::PIECE);
                __syncwarp();
                // Test hook: the first stage's bytes are expected but never copied, so
                // the stage never completes (the barrier phases stay exact).
                if (!(a.fault_mode == 1 && jb == 0 && valid != 0u)) {
                    if (contig) {
                        if (lane == 0) bulk_load(dst, pool + size_t(r0) * row_bytes, C::KV_BYTES, &fullb[st]);
                    } else if (row >= 0) {
                        bulk_load(dst + uint32_t(lane * C::PIECE), pool + size_t(row) * row_bytes, C::PIECE,
                                  &fullb[st]);
                    }
                }
                if (!RANGE && !is_v && blk == w.nblk - 1 && a.gate != nullptr && w.complete) {
                    // the segment's gate rows, read by its epilogue a few blocks from now:
                    // into L2 (two 128-byte lines per row of HB * G rows)
                    for (int x = lane; x < C::HB * a.Mq * 2; x += 32) {
                        const int n = x >> 1, gq = n / a.Mq, r = n % a.Mq;
                        prefetch_l2(a.gate + (((size_t)w.b * a.Sq + r / a.G) * a.Hq + (hb0 + gq) * a.G + r % a.G) *
                                                 C::D + (x & 1) * 64);
                    }
                }
            }
            w.advance();
        }
        if (failed) {
            if (lane == 0) flag_error(a.err, kErrTimeout);
            *abort_flag = 1;
        }
        // Every copy this warp issued lands before the CTA's shared memory is
        // released.  (Each issued block arrived once on its stage, so the last
        // nst blocks are exactly the fills that can still be in flight.)
        if (lane == 0) {
            for (int q = max(0, issued - nst); q < issued; ++q) {
                if (a.fault_mode == 1 && q == 0) continue;  // never completes, has no copies in flight
                if (!mbar_wait_bounded(&fullb[q % nst], (q / nst) & 1, a.wait_limit_ns, nullptr))
                    flag_error(a.err, kErrTimeout);
            }
        }
        return;  // producers never touch TMEM
    }

    if (warp == C::ISSUER) {
        // ============================================================ MMA issuer
        if (lane == 0) {
            const uint32_t idesc_qk = idesc_e4m3_f32(128, C::N, false, false);
            const uint32_t idesc_pv = idesc_e4m3_f32(128, C::N, true, true);
            const uint32_t kring = smem_u32(smem + C::K_OFF);
            const uint32_t vring = smem_u32(smem + C::V_OFF);
            const uint32_t qaddr = smem_u32(smem + C::Q_OFF);
            const uint32_t paddr = smem_u32(smem + C::P_OFF);
            // Two walks over the same blocks: the next score product QK(qj) and the
            // next output product PV(pj < qj).  Whichever is ready is issued, so an
            // output product never waits on a later block's copies and a score
            // product never waits on an earlier block's softmax.
            PagedBlockWalk qw, pw;
            qw.init(w_begin, w_end, seg_b, seg_p, last_worker);
            pw.init(w_begin, w_end, seg_b, seg_p, last_worker);
            bool q_has = qw.next<RANGE>(a);
            if (q_has) pw.next<RANGE>(a);
            int qj = 0, pj = 0;
            bool ok = true;
            uint64_t t_last = globaltimer_ns();
            uint32_t idle = 0;
            while (ok && (q_has || pj < qj)) {
                bool prog = false;
                // the output product first: it frees a V stage and a P buffer
                if (pj < qj) {
                    const int pb = pj % C::P_BUFS, vs = pj % C::VST;
                    const bool first = pw.blk == 0;
                    // a segment's first PV overwrites O: the previous segment's epilogue has read it
                    if (mbar_test_wait(&p_full[pb], (pj / C::P_BUFS) & 1) &&
                        mbar_test_wait(&vfull[vs], (pj / C::VST) & 1) &&
                        (!first || pw.ns == 0 || mbar_test_wait(o_free, (pw.ns - 1) & 1))) {
                        tc_fence_after_sync();
                        const uint32_t vaddr = vring + vs * C::KV_BYTES;
                        const uint32_t pbase = paddr + pb * 2 * C::P_BYTES;
#pragma unroll
                        for (int piece = 0; piece < 2; ++piece)
#pragma unroll
                            for (int kk = 0; kk < 4; ++kk) {  // 32 (token, head) rows per step
                                const uint64_t ad = smem_desc_sw128(vaddr + kk * 4096, 1024, 1024);
                                const uint64_t bd =
                                    smem_desc_plain(pbase + piece * C::P_BYTES + kk * 512, 128, C::P_NBLK);
                                umma_e4m3(tbase + (piece ? C::OL_COL : C::OH_COL), ad, bd, idesc_pv,
                                          (first && kk == 0) ? 0u : 1u);
                            }
                        umma_commit(&pv_done[pb]);
                        umma_commit(&vempty[vs]);
                        ++pj;
                        if (pj < qj || q_has) pw.next<RANGE>(a);
                        prog = true;
                    }
                }
                if (q_has) {
                    const int ks = qj % C::KST;
                    if ((qw.blk != 0 || mbar_test_wait(q_full, qw.ns & 1)) &&
                        mbar_test_wait(&kfull[ks], (qj / C::KST) & 1) &&
                        (qj < 2 || mbar_test_wait(&s_free[qj & 1], ((qj - 2) >> 1) & 1))) {
                        tc_fence_after_sync();
                        const uint32_t kaddr = kring + ks * C::KV_BYTES;
#pragma unroll
                        for (int piece = 0; piece < 2; ++piece)
#pragma unroll
                            for (int kk = 0; kk < 4; ++kk) {  // 32 codes per step
                                const uint64_t ad = smem_desc_sw128(kaddr + kk * 32, 16, 1024);
                                const uint64_t bd = smem_desc_sw128(qaddr + piece * C::Q_BYTES + kk * 32, 16, 1024);
                                umma_e4m3(tbase + C::S_COL + (qj & 1) * C::N, ad, bd, idesc_qk,
                                          (piece | kk) ? 1u : 0u);
                            }
                        umma_commit(&s_full[qj & 1]);
                        umma_commit(&kempty[ks]);
                        ++qj;
                        q_has = qw.next<RANGE>(a);
                        prog = true;
                    }
                }
                if (prog) {
                    t_last = globaltimer_ns();
                    idle = 0;
                } else {
                    // nothing ready: sleep in the barrier instruction (a bounded
                    // suspension) instead of polling, to leave issue slots to the
                    // softmax warp that shares this sub-partition
                    if (pj < qj)
                        mbar_try_wait_for(&p_full[pj % C::P_BUFS], (pj / C::P_BUFS) & 1, 100);
                    else if (q_has)
                        mbar_try_wait_for(&kfull[qj % C::KST], (qj / C::KST) & 1, 100);
                    if ((++idle & 15u) == 0u && (*abort_flag || globaltimer_ns() - t_last > a.wait_limit_ns))
                        ok = false;
                }
            }
            if (!ok) {
                flag_error(a.err, kErrTimeout);
                *abort_flag = 1;
            }
            // drain: every MMA issued has finished before TMEM is freed
            umma_commit(fin);
            mbar_wait_bounded(fin, 0, a.wait_limit_ns, nullptr);
        }
        __syncwarp();
    } else {
        // ============================================================ softmax warps 0-3
        // A wait that runs out poisons this warp: it then skips every wait and
        // tensor-memory access but still takes every named barrier (all 128
        // threads walk the same blocks), so no thread is left in a barrier.
        const int m = threadIdx.x;  // TMEM lane
        const int t = m >> 3;       // token of the block
        const int g = m & 7;        // head of the block
        const uint32_t lane_base = tbase + (uint32_t(warp * 32) << 16);
        const bool causal = RANGE && a.Sq > 1;
        PagedSegWalk w;
        w.init(w_begin, w_end, seg_b, seg_p, last_worker);
        bool failed = false;
        int jb = 0;
        auto wait = [&](uint64_t *bar, uint32_t parity) {
            if (failed) return;
            const bool ok = mbar_wait_bounded(bar, parity, a.wait_limit_ns, abort_flag);
            if (!__all_sync(0xffffffffu, ok)) {
                failed = true;
                *abort_flag = 1;
            }
        };

        // Q' of a segment: row n = g' R + r holds query row r of head hb0 + g',
        // scaled by 2^e (largest element in [128, 256)) and split into E4M3
        // hi / lo pieces, its 16-byte chunks permuted by "xor g'" and stored
        // 128-byte swizzled.  alpha_s[n] = score multiplier of the row.
        auto build_q = [&](const PagedSegWalk &sg) {
            constexpr int TPR = 128 / C::N;  // threads per row
            constexpr int EPT = C::D / TPR;  // elements per thread
            const int n = m / TPR, part = m % TPR;
            const int gq = n / R, r = n % R;
            const bool real = r < a.Mq;
            const int i = real ? r / a.G : 0;
            const int hl = real ? r % a.G : 0;
            const __nv_bfloat16 *qrow =
                a.q + ((size_t(sg.b) * a.Sq + i) * a.Hq + size_t(hb0 + gq) * a.G + hl) * C::D + part * EPT;
            float v[EPT];
            float mx = 0.f;
#pragma unroll
            for (int c = 0; c < EPT / 8; ++c) {
                uint4 raw = make_uint4(0u, 0u, 0u, 0u);
                if (real) raw = *reinterpret_cast<const uint4 *>(qrow + c * 8);
                const uint32_t wv[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    v[c * 8 + 2 * e] = __uint_as_float(wv[e] << 16);
                    v[c * 8 + 2 * e + 1] = __uint_as_float(wv[e] & 0xffff0000u);
                    mx = fmaxf(mx, fmaxf(fabsf(v[c * 8 + 2 * e]), fabsf(v[c * 8 + 2 * e + 1])));
                }
            }
#pragma unroll
            for (int off = 1; off < TPR; off <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
            int ex = mx > 0.f ? 7 - ilogbf(mx) : 0;  // mx * 2^ex in [128, 256)
            ex = ex > 126 ? 126 : ex;
            const float up = ldexpf(1.f, ex);
            uint8_t *qbase = smem + C::Q_OFF;
#pragma unroll
            for (int c = 0; c < EPT / 16; ++c) {
                uint32_t hw[4], lw[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int x = c * 16 + 4 * e;
                    const float a0 = v[x] * up, a1 = v[x + 1] * up, a2 = v[x + 2] * up, a3 = v[x + 3] * up;
                    const uint16_t h01 = f32x2_to_e4m3x2(a0, a1), h23 = f32x2_to_e4m3x2(a2, a3);
                    const float2 f01 = e4m3x2_to_f32x2(h01), f23 = e4m3x2_to_f32x2(h23);
                    const uint16_t l01 = f32x2_to_e4m3x2(a0 - f01.x, a1 - f01.y);
                    const uint16_t l23 = f32x2_to_e4m3x2(a2 - f23.x, a3 - f23.y);
                    hw[e] = uint32_t(h01) | (uint32_t(h23) << 16);
                    lw[e] = uint32_t(l01) | (uint32_t(l23) << 16);
                }
                const int cq = (part * EPT) / 16 + c;  // the query's 16-code chunk
                const int phys = (cq ^ gq) ^ (n & 7);   // logical chunk cq ^ g', swizzled by row
                *reinterpret_cast<uint4 *>(qbase + n * 128 + phys * 16) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
                *reinterpret_cast<uint4 *>(qbase + C::Q_BYTES + n * 128 + phys * 16) =
                    make_uint4(lw[0], lw[1], lw[2], lw[3]);
            }
            if (part == 0) {
                float al = a.alpha;
                if (a.k_scales != nullptr) al *= __ldg(a.k_scales + (a.n_scales > 1 ? hb0 + gq : 0));
                alpha_s[n] = al * ldexpf(1.f, -ex);
            }
            fence_proxy_async_shared();
            softmax_bar();
            if (m == 0 && !failed) mbar_arrive(q_full);
        };
        // Q' of the first non-empty segment after `sg` (or of sg itself)
        auto build_next_q = [&](PagedSegWalk sg, bool skip_current) {
            if (skip_current) sg.advance();
            while (sg.next<RANGE>(a)) {
                if (sg.nblk > 0) {
                    build_q(sg);
                    return;
                }
                sg.advance();
            }
        };
        build_next_q(w, false);

        while (w.next<RANGE>(a)) {
            // per-row state of this thread's head g
            float aw[R], mref[R], l[R];
            int kmax[R];
            const bool nonempty = w.nblk > 0;
#pragma unroll
            for (int r = 0; r < R; ++r) {
                aw[r] = nonempty ? alpha_s[g * R + r] : 0.f;
                mref[r] = -INFINITY;
                l[r] = 0.f;
                kmax[r] = r < a.Mq ? w.seq_len - a.Sq + r / a.G : -1;
            }
            if (m < C::N) {
                mref_s[m] = -INFINITY;
                // where column (g', r) goes: its output row, or its partial row; -1 for padding rows
                const int gq = m / R, r = m % R;
                long long base = -1;
                if (r < a.Mq) {
                    const int i = r / a.G;
                    const int h = (hb0 + gq) * a.G + r % a.G;
                    base = w.complete ? ((long long)(w.b) * a.Sq + i) * a.Hq + h
                                      : (((long long)(hb) * a.num_splits + blockIdx.y) * 2 + w.slot) * C::HB * a.Mq +
                                            gq * a.Mq + r;
                }
                col_base[m] = base;
            }
            softmax_bar();  // col_base is read by every thread from the first block on
            // Gate values of this lane's outputs (top-K form, two bf16 per register),
            // loaded when the segment's last block starts so their latency hides
            // behind that block's work.  (Loading them at the segment's start, to
            // hold them in registers through every block, measured 12 us slower on
            // the 256-request workload.)
            // the gate in the epilogue's layout: 16-byte pieces x = m + 128 i of the
            // segment's output rows (row n = x / 16 holds column n of O^T)
            uint4 graw[RANGE ? 1 : C::OUT_PIECES / 128];
            if constexpr (!RANGE) {
#pragma unroll
                for (int i = 0; i < C::OUT_PIECES / 128; ++i) graw[i] = make_uint4(0u, 0u, 0u, 0u);
            }
            auto load_gate = [&]() {
                if constexpr (!RANGE) {
                    const __nv_bfloat16 *__restrict__ gatep = a.gate;
                    if (gatep != nullptr && w.complete && !failed) {
#pragma unroll
                        for (int i = 0; i < C::OUT_PIECES / 128; ++i) {
                            const int x = m + 128 * i, n = x / (C::D / 8), u = x % (C::D / 8);
                            const long long rb = col_base[n];
                            if (rb >= 0) graw[i] = __ldg(reinterpret_cast<const uint4 *>(gatep + rb * C::D) + u);
                        }
                    }
                }
            };
            if (w.nblk == 0) load_gate();
            for (int blk = 0; blk < w.nblk; ++blk, ++jb) {
                if (blk == w.nblk - 1) load_gate();
                wait(&s_full[jb & 1], (jb >> 1) & 1);
                wait(&vm_full[jb % C::VM_SLOTS], (jb / C::VM_SLOTS) & 1);  // the block's token mask
                // this lane's scores: columns g R .. g R + R - 1 of the N
                float s[R];
#pragma unroll
                for (int r = 0; r < R; ++r) s[r] = 0.f;
                if (!failed) {
                    tc_fence_after_sync();
                    const uint32_t scol = lane_base + C::S_COL + (jb & 1) * C::N;
                    if constexpr (C::N == 16) {
                        uint32_t sr[16];
                        tmem_ld16(scol, sr);
                        tmem_wait_ld();
#pragma unroll
                        for (int r = 0; r < R; ++r) {
                            float v0[4];
#pragma unroll
                            for (int h = 0; h < 4; ++h)
                                v0[h] = __uint_as_float((g & 1) ? sr[(2 * h + 1) * R + r] : sr[(2 * h) * R + r]);
                            const float v1 = (g & 2) ? v0[1] : v0[0], v2 = (g & 2) ? v0[3] : v0[2];
                            s[r] = (g & 4) ? v2 : v1;
                        }
                    } else {
                        // 32 columns per load: four heads of R = 8 (N = 64), all eight of R = 4
#pragma unroll
                        for (int half = 0; half < C::N / 32; ++half) {
                            uint32_t sr[32];
                            tmem_ld32(scol + half * 32, sr);
                            tmem_wait_ld();
                            constexpr int HPL = 32 / R;  // heads per load
#pragma unroll
                            for (int r = 0; r < R; ++r) {
                                float v0[HPL / 2];
#pragma unroll
                                for (int h = 0; h < HPL / 2; ++h)
                                    v0[h] = __uint_as_float((g & 1) ? sr[(2 * h + 1) * R + r] : sr[(2 * h) * R + r]);
                                float sel;
                                if constexpr (HPL == 8) {
                                    const float v1 = (g & 2) ? v0[1] : v0[0], v2 = (g & 2) ? v0[3] : v0[2];
                                    sel = (g & 4) ? v2 : v1;
                                } else {
                                    sel = (g & 2) ? v0[1] : v0[0];
                                }
                                if (C::N == 32 || ((g >> 2) == half)) s[r] = sel;
                            }
                        }
                    }
                }
                tc_fence_before_sync();
                __syncwarp();
                // a warp that gave up stops arriving anywhere: spurious phases would
                // let the other roles reuse buffers that are still in flight
                if (!failed && lane == 0) mbar_arrive(&s_free[jb & 1]);

                const uint32_t vm = failed ? 0u : vmask[jb % C::VM_SLOTS];
                const bool tvalid = (vm >> t) & 1u;
                const int tokn = w.t_begin + blk * C::BT + t;  // token (list entry) of the request
                float x[R];
                bool need = false;
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    bool vis = tvalid && r < a.Mq;
                    if (causal) vis = vis && tokn <= kmax[r];
                    x[r] = vis ? s[r] * aw[r] : -INFINITY;
                    need |= x[r] > mref[r] + C::kLazy;
                }
                // ---- lazy reference maxima (the vote is the same for all 128 threads)
                if (softmax_bar_any(need)) {
                    float *xb = xch + (jb & 1) * 4 * C::N + warp * C::N;
#pragma unroll
                    for (int r = 0; r < R; ++r) {
                        float v = x[r];
                        v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 8));
                        v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 16));
                        if (lane < 8) xb[g * R + r] = v;  // lanes 0-7: g = lane
                    }
                    softmax_bar();
                    if (m < C::N) {
                        const float *xa = xch + (jb & 1) * 4 * C::N;
                        const float bm = fmaxf(fmaxf(xa[m], xa[C::N + m]), fmaxf(xa[2 * C::N + m], xa[3 * C::N + m]));
                        const float mo = mref_s[m];
                        const float mn = bm > mo + C::kLazy ? bm : mo;
                        corr_s[m] = (mn == mo || mo == -INFINITY) ? 1.f : fast_exp2(mo - mn);
                        mref_s[m] = mn;
                    }
                    softmax_bar();
                    bool resc = false;
#pragma unroll
                    for (int r = 0; r < R; ++r) {
                        const float mn = mref_s[g * R + r];
                        if (mn != mref[r]) l[r] *= corr_s[g * R + r];
                        mref[r] = mn;
                    }
                    // O holds earlier blocks of this segment: rescale the columns whose
                    // reference moved, once the previous block's PV has landed
                    if (blk > 0) {
#pragma unroll
                        for (int n0 = 0; n0 < C::N; ++n0) resc |= corr_s[n0] != 1.f;
                    }
                    if (resc) {
                        const int pj = jb - 1;
                        wait(&pv_done[pj % C::P_BUFS], (pj / C::P_BUFS) & 1);
                        if (!failed) {
                            tc_fence_after_sync();
#pragma unroll
                            for (int part = 0; part < 2; ++part)
#pragma unroll
                                for (int c0 = 0; c0 < C::N; c0 += 16) {
                                    uint32_t ov[16];
                                    const uint32_t ocol = lane_base + (part ? C::OL_COL : C::OH_COL) + c0;
                                    tmem_ld16(ocol, ov);
                                    tmem_wait_ld();
#pragma unroll
                                    for (int e = 0; e < 16; ++e)
                                        ov[e] = __float_as_uint(__uint_as_float(ov[e]) * corr_s[c0 + e]);
                                    tmem_st16(ocol, ov);
                                }
                            tmem_wait_st();
                        }
                    }
                }
                // ---- weights, split into E4M3 hi / lo
                float p[R];
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    const float mu = mref[r] == -INFINITY ? 0.f : mref[r];
                    p[r] = fast_exp2(x[r] - mu + C::kPExp);
                    l[r] += p[r];
                }
                constexpr int NW = R <= 4 ? 1 : 2;  // 32-bit words per piece
                uint32_t hw[NW], lw[NW];
#pragma unroll
                for (int k = 0; k < NW; ++k) hw[k] = lw[k] = 0u;
#pragma unroll
                for (int r = 0; r < R; r += 2) {
                    const uint16_t h = f32x2_to_e4m3x2(p[r], p[r + 1]);
                    const float2 hf = e4m3x2_to_f32x2(h);
                    const uint16_t lo = f32x2_to_e4m3x2(16.f * (p[r] - hf.x), 16.f * (p[r + 1] - hf.y));
                    hw[r / 4] |= uint32_t(h) << (16 * ((r / 2) & 1));
                    lw[r / 4] |= uint32_t(lo) << (16 * ((r / 2) & 1));
                }
                // invalid tokens: their V rows in the stage hold stale bytes (maybe
                // NaN codes); zero this token-and-head's row so 0 x NaN cannot
                // occur, once the stage's copies have landed (the stage is then
                // no longer read by the output product of an earlier block)
                if (vm != 0xffffu) {  // the same for all 128 threads
                    const int vs = jb % C::VST;
                    wait(&vfull[vs], (jb / C::VST) & 1);
                    if (!tvalid && !failed) {
                        uint4 *vrow = reinterpret_cast<uint4 *>(smem + C::V_OFF + vs * C::KV_BYTES + t * C::PIECE +
                                                                g * C::D);
#pragma unroll
                        for (int e = 0; e < C::D / 16; ++e) vrow[e] = make_uint4(0u, 0u, 0u, 0u);
                    }
                }
                // P'^T buffer of this block: free once the PV that last read it is done
                const int pb = jb % C::P_BUFS;
                if (jb >= C::P_BUFS) wait(&pv_done[pb], ((jb - C::P_BUFS) / C::P_BUFS) & 1);
                if (!failed) {
                    // row k = m, columns n = g R .. g R + R - 1 (16-column blocks P_NBLK apart)
                    const int n0 = g * R;
                    uint8_t *ph = smem + C::P_OFF + pb * 2 * C::P_BYTES;
                    const int off = (n0 / 16) * C::P_NBLK + t * 128 + g * 16 + (n0 % 16);
                    if constexpr (R == 2) {
                        *reinterpret_cast<uint16_t *>(ph + off) = uint16_t(hw[0]);
                        *reinterpret_cast<uint16_t *>(ph + C::P_BYTES + off) = uint16_t(lw[0]);
                    } else if constexpr (R == 4) {
                        *reinterpret_cast<uint32_t *>(ph + off) = hw[0];
                        *reinterpret_cast<uint32_t *>(ph + C::P_BYTES + off) = lw[0];
                    } else {
                        *reinterpret_cast<uint2 *>(ph + off) = make_uint2(hw[0], hw[NW - 1]);
                        *reinterpret_cast<uint2 *>(ph + C::P_BYTES + off) = make_uint2(lw[0], lw[NW - 1]);
                    }
                }
                fence_proxy_async_shared();
                tc_fence_before_sync();
                __syncwarp();
                if (!failed && lane == 0) mbar_arrive(&p_full[pb]);

                // last block: Q' of the next non-empty segment (this segment's scores
                // are all computed), so its first QK overlaps this epilogue
                if (blk == w.nblk - 1) build_next_q(w, true);
            }

            // ---- epilogue of the segment
            if (nonempty) {
                const int pj = jb - 1;
                wait(&pv_done[pj % C::P_BUFS], (pj / C::P_BUFS) & 1);
                if (!failed) tc_fence_after_sync();
            }
            const bool dead = softmax_bar_any(failed);  // no output from a CTA that gave up
            const bool gated = !RANGE && a.gate != nullptr && w.complete && !dead;
            // row sums of the 16 lanes of each head
            float *ls = lsum + warp * C::N;
#pragma unroll
            for (int r = 0; r < R; ++r) {
                float v = l[r];
                v += __shfl_xor_sync(0xffffffffu, v, 8);
                v += __shfl_xor_sync(0xffffffffu, v, 16);
                if (lane < 8) ls[g * R + r] = v;
            }
            softmax_bar();
            // per column (g', r) once: the normaliser and the LSE
            if (m < C::N && !dead) {
                const int gq = m / R;
                const long long base = col_base[m];
                float f = 0.f;
                if (base >= 0) {
                    const float L = lsum[m] + lsum[C::N + m] + lsum[2 * C::N + m] + lsum[3 * C::N + m];
                    float vs = a.v_scale;
                    if (a.v_scales != nullptr) vs *= __ldg(a.v_scales + (a.n_scales > 1 ? hb0 + gq : 0));
                    f = L > 0.f ? vs / L : 0.f;
                    const float lse2 = L > 0.f ? mref_s[m] - C::kPExp + log2f(L) : -INFINITY;
                    if (w.complete) {
                        if (a.lse != nullptr) {
                            const int r = m % R, i = r / a.G, h = (hb0 + gq) * a.G + r % a.G;
                            a.lse[((size_t)w.b * a.Hq + h) * a.Sq + i] = lse2 * 0.69314718055994530942f;
                        }
                    } else {
                        a.lse_part[base] = lse2;
                    }
                }
                col_f[m] = f;
            }
            softmax_bar();
            // O is staged in fp32, in natural dimension order, over the P buffers
            // (the segment's last PV has completed, and the next P is written by
            // these threads after the epilogue): lane m holds output dimension
            // d = 16 ((m / 16) ^ g') + m % 16 of head g' in every column (g', r) of
            // O^T.  Then every thread writes whole 16-byte pieces of output rows.
            float *__restrict__ stg = reinterpret_cast<float *>(smem + C::P_OFF);
#pragma unroll
            for (int c0 = 0; c0 < C::N; c0 += 16) {
                uint32_t oh[16], ol[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) oh[e] = ol[e] = 0u;
                if (nonempty && !failed) {
                    tmem_ld16(lane_base + C::OH_COL + c0, oh);
                    tmem_ld16(lane_base + C::OL_COL + c0, ol);
                    tmem_wait_ld();
                }
                if (dead) continue;
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const int n = c0 + e;
                    const int d = 16 * ((m >> 4) ^ (n / R)) + (m & 15);
                    stg[n * C::D + d] = (__uint_as_float(oh[e]) + 0.0625f * __uint_as_float(ol[e])) * col_f[n];
                }
            }
            softmax_bar();
            if (!dead) {
                __nv_bfloat16 *__restrict__ outp = a.out;
                float *__restrict__ opart = a.o_part;
#pragma unroll
                for (int i = 0; i < C::OUT_PIECES / 128; ++i) {
                    const int x = m + 128 * i, n = x / (C::D / 8), u = x % (C::D / 8);
                    const long long rb = col_base[n];
                    if (rb < 0) continue;
                    const float4 v0 = *reinterpret_cast<const float4 *>(stg + n * C::D + 8 * u);
                    const float4 v1 = *reinterpret_cast<const float4 *>(stg + n * C::D + 8 * u + 4);
                    float o[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
                    if (w.complete) {
                        if constexpr (!RANGE) {
                            if (gated) {
                                const uint32_t gw[4] = {graw[i].x, graw[i].y, graw[i].z, graw[i].w};
#pragma unroll
                                for (int e = 0; e < 8; ++e) {
                                    const float gv = __uint_as_float((e & 1) ? (gw[e / 2] & 0xffff0000u) : (gw[e / 2] << 16));
                                    o[e] *= __fdividef(1.f, 1.f + __expf(-gv));
                                }
                            }
                        }
                        const uint4 pk = make_uint4(pack_bf16x2(o[0], o[1]), pack_bf16x2(o[2], o[3]),
                                                    pack_bf16x2(o[4], o[5]), pack_bf16x2(o[6], o[7]));
                        *reinterpret_cast<uint4 *>(outp + rb * C::D + 8 * u) = pk;
                    } else {
                        *reinterpret_cast<float4 *>(opart + rb * C::D + 8 * u) = v0;
                        *reinterpret_cast<float4 *>(opart + rb * C::D + 8 * u + 4) = v1;
                    }
                }
            }
            softmax_bar();
            // P'^T's off-diagonal blocks are never written by the softmax: put back
            // the zeros the staging overwrote (before the next block's P is
            // published to the tensor core, which fences the async proxy)
            for (int i = m; i < C::P_BUFS * 2 * C::P_BYTES / 16; i += 128)
                reinterpret_cast<uint4 *>(smem + C::P_OFF)[i] = make_uint4(0u, 0u, 0u, 0u);
            if (nonempty && !failed) {
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(o_free);
            }
            softmax_bar();  // lsum and mref_s are reused by the next segment
            w.advance();
        }
        if (failed && lane == 0) flag_error(a.err, kErrTimeout);
        pdl_launch_dependents();
    }

    // ---- teardown (issuer and softmax warps): all MMAs and TMEM accesses are done; free TMEM
    tc_fence_before_sync();
    asm volatile("bar.sync 2, 160;" ::: "memory");
    if (warp == C::ISSUER) {
        tc_fence_after_sync();
        tmem_dealloc(tbase, C::TMEM_COLS);
    }
}

}  // namespace gqa
