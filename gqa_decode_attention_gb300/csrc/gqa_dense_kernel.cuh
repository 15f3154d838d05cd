// gqa_dense_kernel.cuh -- split-KV grouped-query decode attention (sm_103a).
//
// One CTA owns one (batch row b, KV head g, KV split s) and up to 128 query
// rows of that KV head's group: rows r = i * G + hl (decode row i < Sq, local
// head hl < G = Hq / Hkv, query head h = g * G + hl).  Query head h therefore
// reads KV head g = h / (Hq / Hkv) in place ("When the K/V copy costs more than
// the attention", section "What I was looking at"), and each K/V byte of the
// split is fetched from HBM once for the whole group.
//
// Pipeline: warp 0 is the producer -- one lane issues TMA tile loads
// (cp.async.bulk.tensor, 128-byte swizzle) of K and V into a ring of shared
// memory stages guarded by full / empty mbarriers.  Each consumer warp owns a
// block of 16 query rows and walks every key of the split in order, 16 keys
// per step: S = Q K^T on the tensor cores (bf16 in, fp32 accumulate), the
// bottom-right causal mask, the online softmax in base 2 with the scale folded
// into one multiplier, and O += P V.  A row's arithmetic therefore depends
// only on the split boundaries (multiples of 64 keys) and never on how many
// rows share the CTA, which makes native GQA bit-identical to the same kernel
// run on K/V expanded to every query head.  With one split the CTA writes
// bf16 O and fp32 LSE; otherwise fp32 partials (O / l and log2-domain LSE) for
// the combine kernel.  D is the score head size (q, K) and DV the value head
// size (V, O, partials); they differ only in the d192x128 instance.
//
// Key lanes (KS > 1): the consumer warps form KS key lanes of RB row blocks;
// lane k walks the tiles k, k + KS, k + 2 KS, ... of the CTA's split through
// the same ring with its own online-softmax state, and at the end the lanes'
// (maximum, sum, unnormalised O) are merged in shared memory by lane 0, which
// writes the result (one split: a small cache, or a unit whose CTA fills an
// SM, in one launch without a combine pass) or the split's partials.  The
// flash-decoding split of the KV walk, done inside one CTA.
//
// Every mbarrier wait is bounded in wall time; on expiry the CTA flags the
// device error word, waits (bounded) for its own loads still in flight, and
// returns.
#pragma once

#include "gqa_common.cuh"
#include "gqa_params.h"

namespace gqa {

// Keys per online-softmax step (one m16n8k16 k-group of keys).
constexpr int kStepKeys = 16;

// Shape of one kernel instance: RB consumer warps (16 rows each) per key
// lane, KS key lanes, TMA tiles of T keys, STAGES ring slots.  Chosen per
// (head dim, row count) so small-group CTAs are small and many fit on an SM.
template <int D, int DV, int RB, int T, int STAGES_, int KS = 1>
struct DenseCfg {
    static constexpr int NC = RB * KS;
    static constexpr int THREADS = 32 * (NC + 1);
    static constexpr int STAGES = STAGES_;
    static constexpr int K_CHUNKS = D / 64;   // 128-byte swizzle atoms per K row (D = score head size)
    static constexpr int V_CHUNKS = DV / 64;  // ... per V row (DV = value head size)
    static constexpr int K_TILE_BYTES = T * D * 2;
    static constexpr int V_TILE_BYTES = T * DV * 2;
    static constexpr int STAGE_BYTES = K_TILE_BYTES + V_TILE_BYTES;
    static constexpr int QROWS = RB * 16;
    static constexpr int Q_BYTES = QROWS * D * 2;
    static constexpr int RING_BYTES = STAGES * STAGE_BYTES;
    static constexpr int BAR_OFF = RING_BYTES + Q_BYTES;
    static constexpr int SMEM_BYTES = BAR_OFF + 2 * STAGES * 8 + 16 + 1024;  // +1024 alignment slack
    static constexpr int MIN_BLOCKS_RAW = (227 * 1024) / SMEM_BYTES;
    static constexpr int MIN_BLOCKS = MIN_BLOCKS_RAW < 1 ? 1 : (MIN_BLOCKS_RAW > 8 ? 8 : MIN_BLOCKS_RAW);
    static_assert(kSplitKeys % T == 0 && T % kStepKeys == 0, "tile must divide the split granule");
    // key-lane merge: per lane of every consumer warp, its O fragment (DV / 2
    // floats) and two (maximum, sum) pairs, laid over the drained ring
    static constexpr int MERGE_FLOATS = DV / 2 + 4;
    static_assert(KS == 1 || NC * 32 * MERGE_FLOATS * 4 <= RING_BYTES, "merge area fits the ring");
    // A consumer waits for tile `it` on its stage's full barrier by phase
    // parity, which is unambiguous only if that stage's previous tile
    // (it - STAGES) has landed.  With STAGES a multiple of KS that tile belongs
    // to the same key lane, which consumed it before.  Otherwise a lane running
    // ahead of another could see a phase two back as complete (parity alone
    // cannot tell "tile it - STAGES not landed" from "tile it landed").  So it
    // first waits on the stage's empty barrier for tile it - STAGES to have
    // been consumed (hence landed).  That wait is unambiguous: the producer
    // fills stages in order, so once a lane has consumed tile it - KS every
    // tile up to it - KS - STAGES has been consumed -- with STAGES >= KS that
    // includes it - 2 STAGES -- and tile it has not.
    static constexpr bool TWO_STEP_WAIT = KS > 1 && STAGES % KS != 0;
    static_assert(STAGES >= KS, "ring at least as deep as the key lanes");
};

template <int D, int DV, int RB, int T, int STAGES_, int KS = 1>
__global__ void __launch_bounds__(DenseCfg<D, DV, RB, T, STAGES_, KS>::THREADS,
                                  DenseCfg<D, DV, RB, T, STAGES_, KS>::MIN_BLOCKS)
    gqa_dense_split_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                           const DenseArgs a) {
    using C = DenseCfg<D, DV, RB, T, STAGES_, KS>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *ring = smem;
    uint8_t *qs = smem + C::RING_BYTES;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + C::BAR_OFF);
    uint64_t *empty = full + C::STAGES;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(empty + C::STAGES);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // Grid: x = (KV head, row group) fastest, so the CTAs of one split that
    // stream neighbouring heads of the same keys start together; y = split.
    const int g = blockIdx.x / a.row_groups;
    const int rg = blockIdx.x % a.row_groups;
    const int split = blockIdx.y;
    const int b = blockIdx.z;
    const int key_begin = split * a.blocks_per_split * kSplitKeys;
    const int key_end = min(a.Skv, key_begin + a.blocks_per_split * kSplitKeys);
    const int n_it = (key_end - key_begin + T - 1) / T;

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], RB);  // the row blocks of the tile's key lane
        }
        *abort_flag = 0;
        fence_mbarrier_init();
    }
    __syncthreads();

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            prefetch_tmap(&tmK);
            prefetch_tmap(&tmV);
            int issued = 0;
            bool ok = true;
            for (int it = 0; it < n_it; ++it) {
                const int st = it % C::STAGES;
                const int round = it / C::STAGES;
                if (round > 0 && !mbar_wait_bounded(&empty[st], (round - 1) & 1, a.wait_limit_ns, abort_flag)) {
                    ok = false;
                    break;
                }
                if (a.fault_mode == 1 && it == 0) {
                    issued = 1;
                    continue;  // test hook: this stage never fills
                }
                uint8_t *ks = ring + st * C::STAGE_BYTES;
                uint8_t *vs = ks + C::K_TILE_BYTES;
                const int j0 = key_begin + it * T;
                mbar_arrive_expect_tx(&full[st], C::STAGE_BYTES);
#pragma unroll
                for (int c = 0; c < C::K_CHUNKS; ++c) tma_load_4d(ks + c * T * 128, &tmK, &full[st], c * 64, g, j0, b);
#pragma unroll
                for (int c = 0; c < C::V_CHUNKS; ++c) tma_load_4d(vs + c * T * 128, &tmV, &full[st], c * 64, g, j0, b);
                issued = it + 1;
            }
            if (!ok) {
                flag_error(a.err, kErrTimeout);
                *abort_flag = 1;
            }
            // Never leave the CTA with a copy still landing in shared memory:
            // wait for the last loads issued (those not yet released).
            if (!ok || *abort_flag) {
                for (int it = max(0, issued - C::STAGES); it < issued; ++it) {
                    if (a.fault_mode == 1 && it == 0) continue;
                    mbar_wait_bounded(&full[it % C::STAGES], (it / C::STAGES) & 1, a.wait_limit_ns, nullptr);
                }
            }
        }
        return;
    }

    // ---------------------------------------------------------------- consumers
    const int rb = (warp - 1) % RB;  // row block of this warp
    const int ks = (warp - 1) / RB;  // key lane: tiles ks, ks + KS, ...
    const int cthreads = C::NC * 32;
    const int ctid = threadIdx.x - 32;

    // Stage this CTA's query rows into shared memory (128-byte swizzled,
    // chunk-major like the K/V tiles).  Rows beyond Mq are zero.
    for (int idx = ctid; idx < C::QROWS * (D / 8); idx += cthreads) {
        const int lr = idx / (D / 8);
        const int u = idx % (D / 8);
        const int r = rg * C::QROWS + lr;
        uint4 val = make_uint4(0, 0, 0, 0);
        if (r < a.Mq) {
            const int i = r / a.G;
            const int h = g * a.G + (r % a.G);
            const __nv_bfloat16 *src = a.q + ((size_t(b) * a.Sq + i) * a.Hq + h) * D + u * 8;
            val = *reinterpret_cast<const uint4 *>(src);
        }
        *reinterpret_cast<uint4 *>(qs + (u >> 3) * (C::QROWS * 128) + swz128(lr, u & 7)) = val;
    }
    asm volatile("bar.sync 1, %0;" ::"r"(cthreads) : "memory");

    // Rows held by this thread: local rows rb*16 + lane/4 and +8.
    int kmax[2];
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
        const int r = rg * C::QROWS + rb * 16 + (lane >> 2) + 8 * hr;
        const int i = r < a.Mq ? r / a.G : a.Sq - 1;
        kmax[hr] = a.Skv - a.Sq + i;  // last visible key (bottom-right causal)
    }
    const int mask_from = a.Skv - a.Sq;  // steps ending at or below this key need no mask

    float m_run[2] = {-INFINITY, -INFINITY};
    float l_run[2] = {0.f, 0.f};
    float o[DV / 8][4];
#pragma unroll
    for (int nt = 0; nt < DV / 8; ++nt) o[nt][0] = o[nt][1] = o[nt][2] = o[nt][3] = 0.f;

    const uint32_t q_base = smem_u32(qs);
    const uint32_t ring_base = smem_u32(ring);
    bool failed = false;

    for (int it = ks; it < n_it; it += KS) {
        const int st = it % C::STAGES;
        // ldmatrix / mma.sync are warp-collective: the whole warp leaves together.
        bool got = true;
        if constexpr (C::TWO_STEP_WAIT) {
            if (it >= C::STAGES) got = mbar_wait_bounded(&empty[st], (it / C::STAGES - 1) & 1, a.wait_limit_ns, abort_flag);
        }
        got = got && mbar_wait_bounded(&full[st], (it / C::STAGES) & 1, a.wait_limit_ns, abort_flag);
        if (!__all_sync(0xffffffffu, got)) {
            failed = true;
            break;
        }
        const uint32_t kb = ring_base + st * C::STAGE_BYTES;
        const uint32_t vb = kb + C::K_TILE_BYTES;
#pragma unroll 1
        for (int sub = 0; sub < T / kStepKeys; ++sub) {
            const int krow0 = sub * kStepKeys;  // first key row of this step in the tile
            const int key0 = key_begin + it * T + krow0;
            if (key0 >= a.Skv) break;  // past the cache: a fully masked step is a no-op

            // ---- S = Q K^T for this warp's 16 rows x 16 keys
            float s[2][4];
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                uint32_t af[4];
                {
                    const int unit = kk * 2 + (lane >> 4);
                    const uint32_t addr =
                        q_base + (unit >> 3) * (C::QROWS * 128) + swz128(rb * 16 + (lane & 15), unit & 7);
                    ldsm_x4(addr, af[0], af[1], af[2], af[3]);
                }
                const int unit = kk * 2 + ((lane >> 3) & 1);
                const int krow = krow0 + (lane & 7) + 8 * (lane >> 4);
                const uint32_t addr = kb + (unit >> 3) * (T * 128) + swz128(krow, unit & 7);
                uint32_t b0, b1, b2, b3;
                ldsm_x4(addr, b0, b1, b2, b3);
                mma_bf16_16816(s[0], af, b0, b1);
                mma_bf16_16816(s[1], af, b2, b3);
            }

            // ---- scale into the log2 domain, mask, online softmax
            const bool need_mask = (key0 + kStepKeys - 1) > mask_from;
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    float t = s[nt][e] * a.alpha;
                    if (need_mask) {
                        const int key = key0 + nt * 8 + (lane & 3) * 2 + (e & 1);
                        if (key > kmax[e >> 1]) t = -INFINITY;
                    }
                    s[nt][e] = t;
                }
            float corr[2];
#pragma unroll
            for (int hr = 0; hr < 2; ++hr) {
                float mx = fmaxf(fmaxf(s[0][2 * hr], s[0][2 * hr + 1]), fmaxf(s[1][2 * hr], s[1][2 * hr + 1]));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
                const float m_new = fmaxf(m_run[hr], mx);
                const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
                corr[hr] = fast_exp2(m_run[hr] - m_use);
                m_run[hr] = m_new;
                float psum = 0.f;
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) {
                    s[nt][2 * hr] = fast_exp2(s[nt][2 * hr] - m_use);
                    s[nt][2 * hr + 1] = fast_exp2(s[nt][2 * hr + 1] - m_use);
                    psum += s[nt][2 * hr] + s[nt][2 * hr + 1];
                }
                l_run[hr] = l_run[hr] * corr[hr] + psum;
            }
            // P in bf16 as the A operand of the PV product:
            // a0 (row, k 0-7), a1 (row+8, k 0-7), a2 (row, k 8-15), a3 (row+8, k 8-15)
            const uint32_t pf[4] = {pack_bf16x2(s[0][0], s[0][1]), pack_bf16x2(s[0][2], s[0][3]),
                                    pack_bf16x2(s[1][0], s[1][1]), pack_bf16x2(s[1][2], s[1][3])};
            if (__any_sync(0xffffffffu, corr[0] != 1.f || corr[1] != 1.f)) {
#pragma unroll
                for (int nt = 0; nt < DV / 8; ++nt) {
                    o[nt][0] *= corr[0];
                    o[nt][1] *= corr[0];
                    o[nt][2] *= corr[1];
                    o[nt][3] *= corr[1];
                }
            }

            // ---- O += P V
            const int vrow = krow0 + (lane & 7) + 8 * ((lane >> 3) & 1);
#pragma unroll
            for (int dp = 0; dp < DV / 16; ++dp) {
                const int unit = dp * 2 + (lane >> 4);
                const uint32_t addr = vb + (unit >> 3) * (T * 128) + swz128(vrow, unit & 7);
                uint32_t b0, b1, b2, b3;
                ldsm_x4_t(addr, b0, b1, b2, b3);
                mma_bf16_16816(o[2 * dp], pf, b0, b1);
                mma_bf16_16816(o[2 * dp + 1], pf, b2, b3);
            }
        }

        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[st]);
    }

    if (failed) {
        flag_error(a.err, kErrTimeout);
        *abort_flag = 1;
    }
    pdl_launch_dependents();
    if constexpr (KS == 1) {
        if (failed || *abort_flag) return;
    }

    // ---- row sums across the 4 lanes that share a row
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
        l_run[hr] += __shfl_xor_sync(0xffffffffu, l_run[hr], 1);
        l_run[hr] += __shfl_xor_sync(0xffffffffu, l_run[hr], 2);
    }

    if constexpr (KS > 1) {
        // Every consumer warp gets here (a failed one too), so the barriers below
        // always complete; the decision to write anything is taken after the
        // first one, from the shared abort flag.  Past it every tile has been
        // consumed, so every copy has landed and the ring is free.
        asm volatile("bar.sync 1, %0;" ::"r"(cthreads) : "memory");
        if (*abort_flag) return;
        float *mx = reinterpret_cast<float *>(ring) + size_t((warp - 1) * 32 + lane) * C::MERGE_FLOATS;
#pragma unroll
        for (int nt = 0; nt < DV / 8; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) mx[nt * 4 + e] = o[nt][e];
        mx[DV / 2 + 0] = m_run[0];
        mx[DV / 2 + 1] = m_run[1];
        mx[DV / 2 + 2] = l_run[0];
        mx[DV / 2 + 3] = l_run[1];
        asm volatile("bar.sync 1, %0;" ::"r"(cthreads) : "memory");
        if (ks != 0) return;
        // lane 0 merges lanes 0 .. KS-1 of its row block, in lane order:
        // M = max m_k, O = sum 2^(m_k - M) O_k, L = sum 2^(m_k - M) l_k
        const float *base = reinterpret_cast<const float *>(ring);
        float mk[KS][2];
#pragma unroll
        for (int k = 0; k < KS; ++k) {
            const float *src = base + size_t((k * RB + rb) * 32 + lane) * C::MERGE_FLOATS;
            mk[k][0] = src[DV / 2 + 0];
            mk[k][1] = src[DV / 2 + 1];
        }
        float wk[KS][2];
#pragma unroll
        for (int hr = 0; hr < 2; ++hr) {
            float M = mk[0][hr];
#pragma unroll
            for (int k = 1; k < KS; ++k) M = fmaxf(M, mk[k][hr]);
            const float M_use = (M == -INFINITY) ? 0.f : M;
#pragma unroll
            for (int k = 0; k < KS; ++k) wk[k][hr] = (mk[k][hr] == -INFINITY) ? 0.f : fast_exp2(mk[k][hr] - M_use);
            m_run[hr] = M;
            l_run[hr] = 0.f;
        }
#pragma unroll
        for (int nt = 0; nt < DV / 8; ++nt) o[nt][0] = o[nt][1] = o[nt][2] = o[nt][3] = 0.f;
#pragma unroll
        for (int k = 0; k < KS; ++k) {
            const float *src = base + size_t((k * RB + rb) * 32 + lane) * C::MERGE_FLOATS;
            l_run[0] += wk[k][0] * src[DV / 2 + 2];
            l_run[1] += wk[k][1] * src[DV / 2 + 3];
#pragma unroll
            for (int nt = 0; nt < DV / 8; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) o[nt][e] += wk[k][e >> 1] * src[nt * 4 + e];
        }
    }

    // ---- epilogue
    const int unit = b * a.Hkv + g;
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
        const int r = rg * C::QROWS + rb * 16 + (lane >> 2) + 8 * hr;
        if (r >= a.Mq) continue;
        const float L = l_run[hr];
        const float inv = L > 0.f ? 1.f / L : 0.f;
        const float lse2 = L > 0.f ? m_run[hr] + log2f(L) : -INFINITY;
        const int i = r / a.G;
        const int h = g * a.G + (r % a.G);
        if (a.num_splits == 1) {
            __nv_bfloat16 *dst = a.out + ((size_t(b) * a.Sq + i) * a.Hq + h) * DV + (lane & 3) * 2;
#pragma unroll
            for (int nt = 0; nt < DV / 8; ++nt)
                *reinterpret_cast<uint32_t *>(dst + nt * 8) =
                    pack_bf16x2(o[nt][2 * hr] * inv, o[nt][2 * hr + 1] * inv);
            if (a.lse != nullptr && (lane & 3) == 0)
                a.lse[(size_t(b) * a.Hq + h) * a.Sq + i] = lse2 * 0.69314718055994530942f;
        } else {
            const size_t prow = (size_t(unit) * a.Mq + r) * a.num_splits + split;
            float *dst = a.o_part + prow * DV + (lane & 3) * 2;
#pragma unroll
            for (int nt = 0; nt < DV / 8; ++nt)
                *reinterpret_cast<float2 *>(dst + nt * 8) = make_float2(o[nt][2 * hr] * inv, o[nt][2 * hr + 1] * inv);
            if ((lane & 3) == 0) a.lse_part[prow] = lse2;
        }
    }
}

// LSE-weighted combine of the split partials.  One CTA per output row
// (b, h, i): the split LSEs give weights w_s = 2^(lse_s - max) (a split that
// saw no visible key has lse_s = -inf and weight exactly 0), and
// O = sum_s w_s O_s / sum_s w_s.  The kernel is latency-bound (a few KiB per
// row, read from L2), so it is laid out for few dependent round trips: every
// thread first starts asynchronous copies of all its partial rows into shared
// memory (no registers held), each warp then reduces the row maximum and the
// weight sum over all splits by itself (shuffles, no block barrier), and the
// only block-wide step is the final sum across the threads that hold
// different splits of the same head-dim values.  The first SC splits are
// staged; any beyond that (very long caches) are read directly.
constexpr int kCombineThreads = 256;
constexpr int kCombineStageBytes = 44 * 1024;  // staged partial rows per CTA (with the sums: <= 48 KiB)

template <int D>
__host__ __device__ constexpr int combine_staged_splits(int S) {
    return S < kCombineStageBytes / (D * 4) ? S : kCombineStageBytes / (D * 4);
}

template <int D>
__global__ void __launch_bounds__(kCombineThreads) gqa_combine_kernel(const float *__restrict__ o_part,
                                                                      const float *__restrict__ lse_part,
                                                                      __nv_bfloat16 *out, float *lse, int Sq,
                                                                      int Hq, int Hkv, int G, int Mq, int S) {
    constexpr int C4 = D / 4;                 // float4 chunks per row
    constexpr int SL = kCombineThreads / C4;  // split lanes
    extern __shared__ float4 cmb_smem[];      // [SC][C4] staged partial rows, then [SL][C4] sums
    const int SC = combine_staged_splits<D>(S);
    float4 *stage = cmb_smem;
    float4 *red = cmb_smem + size_t(SC) * C4;

    pdl_wait_primary();
    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const long row = blockIdx.x;  // (unit * Mq + r)
    const int r = int(row % Mq);
    const long unit = row / Mq;
    const int g = int(unit % Hkv);
    const int b = int(unit / Hkv);
    const float *lp = lse_part + size_t(row) * S;
    const float *op = o_part + size_t(row) * S * D;
    const int c = tid % C4;
    const int sl = tid / C4;

    // 1. this thread's splits s = sl + k SL: copies of the partial rows in flight
    for (int s = sl; s < SC; s += SL) cp_async16(stage + s * C4 + c, op + size_t(s) * D + c * 4);

    // 2. row maximum and weight sum over all splits, per warp
    float M = -INFINITY;
    for (int s = lane; s < S; s += 32) M = fmaxf(M, __ldg(lp + s));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    const float Mu = (M == -INFINITY) ? 0.f : M;
    float L = 0.f;
    for (int s = lane; s < S; s += 32) {
        const float l2 = __ldg(lp + s);
        L += (l2 == -INFINITY) ? 0.f : fast_exp2(l2 - Mu);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) L += __shfl_xor_sync(0xffffffffu, L, off);

    // 3. weighted sum over this thread's splits for its 4 head-dim values
    cp_async_wait_all();
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s = sl; s < S; s += SL) {
        const float l2 = __ldg(lp + s);
        const float w = (l2 == -INFINITY) ? 0.f : fast_exp2(l2 - Mu);
        const float4 x = s < SC ? stage[s * C4 + c] : __ldg(reinterpret_cast<const float4 *>(op + size_t(s) * D) + c);
        acc.x += w * x.x;
        acc.y += w * x.y;
        acc.z += w * x.z;
        acc.w += w * x.w;
    }
    red[tid] = acc;
    __syncthreads();
    if (sl != 0) return;
#pragma unroll
    for (int k = 1; k < SL; ++k) {
        const float4 y = red[k * C4 + c];
        acc.x += y.x;
        acc.y += y.y;
        acc.z += y.z;
        acc.w += y.w;
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;
    const int i = r / G;
    const int h = g * G + (r % G);
    __nv_bfloat16 *dst = out + ((size_t(b) * Sq + i) * Hq + h) * D + c * 4;
    *reinterpret_cast<uint2 *>(dst) = make_uint2(pack_bf16x2(acc.x * inv, acc.y * inv), pack_bf16x2(acc.z * inv, acc.w * inv));
    if (lse != nullptr && c == 0)
        lse[(size_t(b) * Hq + h) * Sq + i] = L > 0.f ? (M + log2f(L)) * 0.69314718055994530942f : -INFINITY;
}

}  // namespace gqa
