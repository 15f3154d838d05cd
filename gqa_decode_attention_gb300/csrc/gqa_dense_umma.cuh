// gqa_dense_umma.cuh -- split-KV grouped-query decode on the fifth-generation
// tensor cores (tcgen05 + TMEM): head dim 256 at every size, and head dim 128
// when a call has many decode rows per head (the contractions then no longer
// fit the legacy tensor pipe's latency budget).
//
// Same unit of work as the mma.sync kernel: one CTA owns (batch row b, KV
// head g, KV split s) and up to 128 query rows of that head's group (rows
// r = i * G + hl, h = g * G + hl), so query head h reads KV head
// g = h / (Hq / Hkv) in place ("When the K/V copy costs more than the
// attention", section "What I was looking at") and each K/V byte of the split
// is read from HBM once for the whole group.
//
// Roles (8 warps):
//   warp 0      TMA producer: K and V tiles of 64 keys x D into a ring of
//               shared-memory stages (128-byte swizzle), full / empty mbarriers.
//   warps 1, 2  leave at once (they keep the issuer off sub-partition 1).
//   warp 3      allocates TMEM; lane 0 issues every MMA:
//                 S(j) = Q K(j)^T   M=128 rows, N=64 keys, K=D  -> TMEM S[j%2]
//                 O   += P(j) V(j)  M=128 rows, N=D,  K=64 keys -> TMEM O
//               so the tensor core computes the next scores while the softmax
//               runs: at D = 128, QK(0), QK(1), then QK(j+2), PV(j) once P(j)
//               is out; at D = 256, PV(j) once P(j) is out and QK(j+1) as soon
//               as its tile lands.
//   warps 4..7  one thread per query row (TMEM lane): load the S row, take
//               the maximum, causal mask, online softmax in the log2 domain,
//               write P(j) as bf16 to shared-memory buffer j % NP (the A
//               operand of PV), and the epilogue.
// The online softmax keeps a per-row reference maximum and rescales O (in
// TMEM) only when a row's maximum grows by more than 2^8; in between, the
// weights are exp2(s - reference) <= 2^8, which changes rounding only.  Every
// row is processed by its own thread with the same instruction sequence, so
// a row's result never depends on how many rows share the CTA.
//
// Every wait is bounded in wall time; on expiry the CTA flags the device
// error word, drains its own copies and MMAs, frees its TMEM and returns.
#pragma once

#include "gqa_common.cuh"
#include "gqa_params.h"
#include "gqa_umma.cuh"

namespace gqa {

// Longest suspension of the MMA issuer in one wait on P while the next tile's
// scores are still to be issued (nanoseconds).
#ifndef GQA_UMMA_ISSUER_POLL_NS
#define GQA_UMMA_ISSUER_POLL_NS 200
#endif
constexpr uint32_t kIssuerPollNs = GQA_UMMA_ISSUER_POLL_NS;

// Whether the producer waits for Q in TMEM after requesting tile 0 (1) or
// requests the whole ring at once (0); a compile-time knob for tuning builds.
#ifndef GQA_UMMA_Q_BEFORE_RING
#define GQA_UMMA_Q_BEFORE_RING 1
#endif

// Keys per tile of the tcgen05 engine; a compile-time knob for tuning builds.
#ifndef GQA_UMMA_TILE_KEYS
#define GQA_UMMA_TILE_KEYS 64
#endif

template <int D>
struct UmmaCfg {
    static constexpr int BM = 128;                  // query rows per CTA (TMEM lanes)
    static constexpr int BN = GQA_UMMA_TILE_KEYS;   // keys per tile (32 or 64)
    static constexpr int CHUNKS = D / 64;
    static constexpr int TILE_BYTES = BN * D * 2;  // K or V tile
    static constexpr int STAGE_BYTES = 2 * TILE_BYTES;
    // Order of the two products once P(j) is out.  A score product is a
    // chain of D / 16 dependent MMAs (about 150 clocks a step on GB300,
    // whatever N is), and S(j+2) is what the softmax waits for next, so at
    // D = 128 QK(j+2) is issued ahead of PV(j) and runs first in the tensor
    // pipe.  P(j+2) then no longer waits for PV(j) through the score commit,
    // so P gets a third buffer; and P lives in TMEM (the A operand of PV read
    // from tensor memory), which takes its writes and reads off the shared
    // memory the tiles stream through.  At D = 256 TMEM is full (scores,
    // output and queries) and the tile's bytes dominate: P stays in shared
    // memory, PV(j) goes first, then QK(j+1) as soon as its tile lands.
#ifndef GQA_UMMA_QK_FIRST
#define GQA_UMMA_QK_FIRST (D == 128)
#endif
    static constexpr bool QK_FIRST = GQA_UMMA_QK_FIRST;
    static constexpr bool P_TMEM = QK_FIRST;         // P in tensor memory
    static constexpr int NP = QK_FIRST ? 3 : 2;      // P buffers
    static constexpr int P_BYTES = BM * 128;  // a shared-memory P buffer: one 128-byte swizzle row a row (BN <= 64)
    static constexpr int NP_SMEM = P_TMEM ? 0 : NP;
    static constexpr int BUDGET = 227 * 1024 - 1024 - 256;
    static constexpr int STAGES_FIT = (BUDGET - NP_SMEM * P_BYTES) / STAGE_BYTES;
#ifndef GQA_UMMA_MAX_STAGES
#define GQA_UMMA_MAX_STAGES 5
#endif
    static constexpr int STAGES = STAGES_FIT > GQA_UMMA_MAX_STAGES ? GQA_UMMA_MAX_STAGES : STAGES_FIT;
    static constexpr int RING_OFF = 0;
    static constexpr int P_OFF = RING_OFF + STAGES * STAGE_BYTES;
    static constexpr int BAR_OFF = P_OFF + NP_SMEM * P_BYTES;
    static constexpr int SMEM_BYTES = BAR_OFF + 256 + 1024;
    // Warp roles: 0 TMA producer, 1 and 2 leave at once, 3 allocates TMEM and
    // issues the MMAs, 4..7 softmax (warp w reads TMEM lane quarter w % 4).
    // The issuer shares SM sub-partition 3 with the softmax warp of lanes
    // 96..127, which hold query rows only when a CTA has more than 96 of
    // them: with the issuer beside a busy softmax warp, every MMA issue waits
    // for issue slots and the score / output chain stretches (measured: 64
    // rows per CTA at d128 ran at 67% of the HBM copy rate with the issuer in
    // sub-partition 1, next to the rows 32..63, and at 80% in sub-partition 3).
    static constexpr int ISSUER = 3;
    static constexpr int SW0 = ISSUER + 1;  // first softmax warp
    static constexpr int THREADS = 32 * SW0 + 128;
    static constexpr uint32_t S_COL = 0;            // two BN-column score buffers
    static constexpr uint32_t O_COL = 2 * BN;       // D columns of fp32 output
    static constexpr uint32_t Q_COL = O_COL + D;    // the CTA's queries, D/2 columns (A operand of QK)
    static constexpr uint32_t P_COL = Q_COL + D / 2;  // P buffers in TMEM, BN/2 columns each (A operand of PV)
    static constexpr uint32_t COLS_USED = P_COL + (P_TMEM ? NP * BN / 2 : 0);
    static constexpr uint32_t TMEM_COLS = COLS_USED <= 256 ? 256 : 512;
    static_assert(COLS_USED <= 512, "TMEM budget");
#ifndef GQA_UMMA_RESCALE_LOG2
#define GQA_UMMA_RESCALE_LOG2 8.f
#endif
    static constexpr float kRescaleLog2 = GQA_UMMA_RESCALE_LOG2;
    static_assert(STAGES >= 3, "QK(j+2) and PV(j) need their tiles in the ring together");
    static_assert(BN == 32 || BN == 64, "tile keys");
    static_assert(D % 64 == 0 && D <= 256, "head dim");
};

template <int D>
__global__ void __launch_bounds__(UmmaCfg<D>::THREADS, 1)
    gqa_dense_umma_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                          const DenseArgs a) {
    using C = UmmaCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *ring = smem + C::RING_OFF;
    uint8_t *ps = smem + C::P_OFF;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + C::BAR_OFF);
    uint64_t *empty = full + C::STAGES;
    uint64_t *s_full = empty + C::STAGES;  // [2]
    uint64_t *p_ready = s_full + 2;        // [2]
    uint64_t *o_done = p_ready + 2;        // [2]: PV(j) completes phase j / 2 of o_done[j % 2]
    uint64_t *fin = o_done + 2;            // [1]
    uint64_t *q_ready = fin + 1;           // [1]
    uint32_t *tmem_base_s = reinterpret_cast<uint32_t *>(q_ready + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_base_s + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int g = blockIdx.x / a.row_groups;
    const int rg = blockIdx.x % a.row_groups;
    const int split = blockIdx.y;
    const int b = blockIdx.z;
    const int key_begin = split * a.blocks_per_split * kSplitKeys;
    const int key_end = min(a.Skv, key_begin + a.blocks_per_split * kSplitKeys);
    const int n_it = (key_end - key_begin + C::BN - 1) / C::BN;

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(&s_full[s], 1);
            mbar_init(&p_ready[s], 128);
            mbar_init(&o_done[s], 1);
        }
        mbar_init(fin, 1);
        mbar_init(q_ready, 128);
        *abort_flag = 0;
        fence_mbarrier_init();
    }
    if (warp == C::ISSUER) tmem_alloc(tmem_base_s, C::TMEM_COLS);
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tbase = *tmem_base_s;

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
                // Tile 0 first, then the query rows: every SM starts by asking for
                // its whole ring at once, and the row threads' plain loads of Q
                // would queue behind all of it, delaying the first scores by
                // microseconds; the rest of the ring is requested once Q is in TMEM.
                if (GQA_UMMA_Q_BEFORE_RING && it == 1 &&
                    !mbar_wait_bounded(q_ready, 0, a.wait_limit_ns, abort_flag)) {
                    ok = false;
                    break;
                }
                if (round > 0 && !mbar_wait_bounded(&empty[st], (round - 1) & 1, a.wait_limit_ns, abort_flag)) {
                    ok = false;
                    break;
                }
                if (a.fault_mode == 1 && it == 0) {
                    issued = 1;
                    continue;  // test hook: this stage never fills
                }
                uint8_t *ks = ring + st * C::STAGE_BYTES;
                uint8_t *vs = ks + C::TILE_BYTES;
                const int j0 = key_begin + it * C::BN;
                mbar_arrive_expect_tx(&full[st], C::STAGE_BYTES);
#pragma unroll
                for (int c = 0; c < C::CHUNKS; ++c)
                    tma_load_4d(ks + c * C::BN * 128, &tmK, &full[st], c * 64, g, j0, b);
#pragma unroll
                for (int c = 0; c < C::CHUNKS; ++c)
                    tma_load_4d(vs + c * C::BN * 128, &tmV, &full[st], c * 64, g, j0, b);
                issued = it + 1;
            }
            if (!ok) {
                flag_error(a.err, kErrTimeout);
                *abort_flag = 1;
            }
            if (!ok || *abort_flag) {
                for (int it = max(0, issued - C::STAGES); it < issued; ++it) {
                    if (a.fault_mode == 1 && it == 0) continue;
                    mbar_wait_bounded(&full[it % C::STAGES], (it / C::STAGES) & 1, a.wait_limit_ns, nullptr);
                }
            }
        }
        return;  // the producer never touches TMEM
    }
    if (warp < C::ISSUER) return;  // spare warps

    if (warp == C::ISSUER) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t idesc_qk = idesc_bf16_f32(C::BM, C::BN, false, false);
            const uint32_t idesc_pv = idesc_bf16_f32(C::BM, D, false, true);
            const uint32_t ring_addr = smem_u32(ring);
            const uint32_t p_addr = smem_u32(ps);
            bool ok = true;
            // QK(j): the tile must have landed, and S[j % 2] is free once the row
            // threads have released P(j - 2) (they read S(j - 2) first).
            auto issue_qk = [&](int j) {
                const int st = j % C::STAGES;
                tc_fence_after_sync();
                const uint32_t kaddr = ring_addr + st * C::STAGE_BYTES;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint64_t bd = smem_desc_sw128(kaddr + (kk >> 2) * (C::BN * 128) + (kk & 3) * 32, 16, 1024);
                    umma_bf16_ta(tbase + C::S_COL + (j & 1) * C::BN, tbase + C::Q_COL + kk * 8, bd, idesc_qk,
                                 kk > 0 ? 1u : 0u);
                }
                umma_commit(&s_full[j & 1]);
            };
            int qk_issued = 0;  // QK(0 .. qk_issued-1) have been issued
            ok = mbar_wait_bounded(q_ready, 0, a.wait_limit_ns, abort_flag);  // Q is in TMEM
            if (ok && n_it > 0) {
                ok = mbar_wait_bounded(&full[0], 0, a.wait_limit_ns, abort_flag);
                if (ok) {
                    issue_qk(0);
                    qk_issued = 1;
                }
            }
            if (C::QK_FIRST && ok && n_it > 1) {
                ok = mbar_wait_bounded(&full[1], 0, a.wait_limit_ns, abort_flag);
                if (ok) {
                    issue_qk(1);
                    qk_issued = 2;
                }
            }
            for (int j = 0; ok && j < n_it; ++j) {
                if (C::QK_FIRST) {
                    // Wait for P(j) (suspended in the barrier instruction), then QK(j+2)
                    // into the score buffer P(j) released -- ahead of PV(j) when its
                    // tile is in, right after it otherwise.
                    const uint64_t t0 = globaltimer_ns();
                    for (uint32_t spin = 1;; ++spin) {
                        if (mbar_try_wait(&p_ready[j & 1], (j >> 1) & 1)) break;
                        if ((spin & 63u) == 0u && (*abort_flag || globaltimer_ns() - t0 > a.wait_limit_ns)) {
                            ok = false;
                            break;
                        }
                    }
                    if (!ok) break;
                    tc_fence_after_sync();
                    const int nx = j + 2;
                    if (nx < n_it && mbar_test_wait(&full[nx % C::STAGES], (nx / C::STAGES) & 1)) {
                        issue_qk(nx);
                        qk_issued = nx + 1;
                    }
                    const int st = j % C::STAGES;
                    const uint32_t vaddr = ring_addr + st * C::STAGE_BYTES + C::TILE_BYTES;
                    const uint32_t pcol = C::P_COL + (j % C::NP) * (C::BN / 2);
#pragma unroll
                    for (int kg = 0; kg < C::BN / 16; ++kg) {
                        const uint64_t bd = smem_desc_sw128(vaddr + kg * 2048, C::BN * 128, 1024);
                        if constexpr (C::P_TMEM) {
                            umma_bf16_ta(tbase + C::O_COL, tbase + pcol + kg * 8, bd, idesc_pv, (j > 0 || kg > 0) ? 1u : 0u);
                        } else {
                            const uint64_t ad =
                                smem_desc_sw128(p_addr + (j % C::NP) * C::P_BYTES + kg * 32, 16, 1024);
                            umma_bf16(tbase + C::O_COL, ad, bd, idesc_pv, (j > 0 || kg > 0) ? 1u : 0u);
                        }
                    }
                    umma_commit(&o_done[j & 1]);
                    umma_commit(&empty[st]);
                    if (nx < n_it && qk_issued == nx) {
                        if (!mbar_wait_bounded(&full[nx % C::STAGES], (nx / C::STAGES) & 1, a.wait_limit_ns,
                                               abort_flag)) {
                            ok = false;
                            break;
                        }
                        issue_qk(nx);
                        qk_issued = nx + 1;
                    }
                    continue;
                }
                // Wait for P(j) while issuing QK(j+1) the moment its tile lands,
                // so PV(j) never waits on the next tile's copy.  The wait on P(j)
                // suspends the thread in the barrier instruction instead of
                // polling: this warp shares an SM sub-partition with softmax warps
                // and must not take their issue slots.  While QK(j+1) is still
                // pending the suspension is capped so the tile is seen soon.
                const uint64_t t0 = globaltimer_ns();
                for (uint32_t spin = 1;; ++spin) {
                    if (qk_issued == j + 1 && j + 1 < n_it &&
                        mbar_test_wait(&full[(j + 1) % C::STAGES], ((j + 1) / C::STAGES) & 1)) {
                        issue_qk(j + 1);
                        qk_issued = j + 2;
                    }
                    const bool pending = qk_issued == j + 1 && j + 1 < n_it;
                    if (pending ? mbar_try_wait_for(&p_ready[j & 1], (j >> 1) & 1, kIssuerPollNs)
                                : mbar_try_wait(&p_ready[j & 1], (j >> 1) & 1))
                        break;
                    if ((spin & 63u) == 0u && (*abort_flag || globaltimer_ns() - t0 > a.wait_limit_ns)) {
                        ok = false;
                        break;
                    }
                }
                if (!ok) break;
                tc_fence_after_sync();
                const int st = j % C::STAGES;
                const uint32_t vaddr = ring_addr + st * C::STAGE_BYTES + C::TILE_BYTES;
                const uint32_t paddr = p_addr + (j & 1) * C::P_BYTES;
#pragma unroll
                for (int kg = 0; kg < C::BN / 16; ++kg) {
                    const uint64_t ad = smem_desc_sw128(paddr + kg * 32, 16, 1024);
                    const uint64_t bd = smem_desc_sw128(vaddr + kg * 2048, C::BN * 128, 1024);
                    umma_bf16(tbase + C::O_COL, ad, bd, idesc_pv, (j > 0 || kg > 0) ? 1u : 0u);
                }
                umma_commit(&o_done[j & 1]);
                umma_commit(&empty[st]);
                if (qk_issued == j + 1 && j + 1 < n_it) {
                    // the next tile was not in yet while P(j) was produced
                    if (!mbar_wait_bounded(&full[(j + 1) % C::STAGES], ((j + 1) / C::STAGES) & 1, a.wait_limit_ns,
                                           abort_flag)) {
                        ok = false;
                        break;
                    }
                    issue_qk(j + 1);
                    qk_issued = j + 2;
                }
            }
            if (!ok) {
                flag_error(a.err, kErrTimeout);
                *abort_flag = 1;
            }
            // Drain: every MMA this thread issued has finished before TMEM is freed.
            umma_commit(fin);
            mbar_wait_bounded(fin, 0, a.wait_limit_ns, nullptr);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ softmax warps
        const int quarter = warp & 3;           // TMEM lane quarter this warp may access
        const int lr = quarter * 32 + lane;     // local row = TMEM lane
        const int r = rg * C::BM + lr;
        const int i_row = r < a.Mq ? r / a.G : a.Sq - 1;
        const int kmax = a.Skv - a.Sq + i_row;  // last visible key (bottom-right causal)
        const int mask_from = a.Skv - a.Sq;
        const uint32_t lane_base = tbase + (uint32_t(quarter * 32) << 16);
        // A warp whose 32 rows all lie past the group's rows only keeps the
        // barrier protocol (its lanes' P rows and O rows are never read out).
        const bool idle = rg * C::BM + quarter * 32 >= a.Mq;
        // This thread's query row -> its TMEM lane, columns Q_COL.. (zeros past Mq).
        {
            const __nv_bfloat16 *qrow =
                a.q + ((size_t(b) * a.Sq + i_row) * a.Hq + g * a.G + (r < a.Mq ? r % a.G : 0)) * D;
#pragma unroll 1
            for (int c = 0; c < D / 64; ++c) {
                uint32_t qv[32];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const uint4 x = r < a.Mq ? *reinterpret_cast<const uint4 *>(qrow + c * 64 + e * 8)
                                             : make_uint4(0, 0, 0, 0);
                    qv[4 * e] = x.x;
                    qv[4 * e + 1] = x.y;
                    qv[4 * e + 2] = x.z;
                    qv[4 * e + 3] = x.w;
                }
                tmem_st32(lane_base + C::Q_COL + c * 32, qv);
            }
            tmem_wait_st();
            tc_fence_before_sync();
            mbar_arrive(q_ready);
        }
        float m_ref = -INFINITY;  // reference maximum (log2 domain)
        float l = 0.f;
        bool failed = false;
        uint8_t *prow_base = ps + lr * 128;

        // tcgen05.ld / st are warp-collective: every TMEM access below is made
        // by all 32 lanes together; per-row conditions only select values and
        // guard the global stores.
        for (int j = 0; j < n_it; ++j) {
            const int sb = j & 1;
            const bool got = mbar_wait_bounded(&s_full[sb], (j >> 1) & 1, a.wait_limit_ns, abort_flag);
            if (!__all_sync(0xffffffffu, got)) {
                failed = true;
                break;
            }
            if (!idle) {
                tc_fence_after_sync();
                uint32_t sr[C::BN / 32][32];
#pragma unroll
                for (int h = 0; h < C::BN / 32; ++h) tmem_ld32(lane_base + C::S_COL + sb * C::BN + h * 32, sr[h]);
                tmem_wait_ld();

                // Scores stay raw; the scale (log2 domain) enters through the
                // maximum (exact: the scale is positive) and one fma per weight.
                const int key0 = key_begin + j * C::BN;
                if (key0 + C::BN - 1 > mask_from) {  // the tile reaches past some row's last visible key
#pragma unroll
                    for (int h = 0; h < C::BN / 32; ++h)
#pragma unroll
                        for (int c = 0; c < 32; ++c)
                            if (key0 + h * 32 + c > kmax) sr[h][c] = __float_as_uint(-INFINITY);
                }
                // the maximum over four independent chains of three-input maxima (exact)
                float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
                for (int h = 0; h < C::BN / 32; ++h)
#pragma unroll
                    for (int c = 0; c < 32; c += 2)
                        m4[(c >> 1) & 3] =
                            fmax3(m4[(c >> 1) & 3], __uint_as_float(sr[h][c]), __uint_as_float(sr[h][c + 1]));
                const float mx = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3])) * a.alpha;
                // A row whose maximum grew by more than 2^8 takes it as the new
                // reference; if it had accumulated anything, its O row is rescaled.
                const bool renew = mx > m_ref + C::kRescaleLog2;
                const bool rescale = renew && l > 0.f;
                if (__any_sync(0xffffffffu, rescale)) {
                    // PV(j-1) must have finished writing O: phase (j-1) / 2 of
                    // o_done[(j-1) % 2].  Unambiguous: S(j) was committed after QK(j),
                    // which was issued after PV(j-3) (after PV(j-2) when PV goes
                    // first), so that barrier's previous phase is complete, and its
                    // next one (PV(j+1)) needs a P this thread has not written yet.
                    const bool od = mbar_wait_bounded(&o_done[(j - 1) & 1], ((j - 1) >> 1) & 1, a.wait_limit_ns,
                                                      abort_flag);
                    if (!__all_sync(0xffffffffu, od)) {
                        failed = true;
                        break;
                    }
                    tc_fence_after_sync();
                    const float corr = rescale ? fast_exp2(m_ref - mx) : 1.f;
#pragma unroll 1
                    for (int c = 0; c < D / 32; ++c) {
                        uint32_t ov[32];
                        tmem_ld32(lane_base + C::O_COL + c * 32, ov);
                        tmem_wait_ld();
#pragma unroll
                        for (int e = 0; e < 32; e += 2) {
                            const float2 o2 = mul2(make_float2(__uint_as_float(ov[e]), __uint_as_float(ov[e + 1])),
                                                   make_float2(corr, corr));
                            ov[e] = __float_as_uint(o2.x);
                            ov[e + 1] = __float_as_uint(o2.y);
                        }
                        tmem_st32(lane_base + C::O_COL + c * 32, ov);
                    }
                    tmem_wait_st();
                    l *= corr;
                }
                if (renew) m_ref = mx;
                const float m_use = (m_ref == -INFINITY) ? 0.f : m_ref;
                // P = exp2(scale * s - reference) as bf16, straight into the swizzled P tile
                // P(j) goes to buffer j % NP, last read by PV(j - NP), which is
                // complete: S(j)'s commit followed QK(j), issued after PV(j - NP).
                // weights exp2(scale * s - reference) for two keys at a time (the
                // two-lane fma rounds each lane as fmaf), summed in two two-lane chains
                const float2 al2 = make_float2(a.alpha, a.alpha), nm2 = make_float2(-m_use, -m_use);
                float2 ps2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
                if constexpr (C::P_TMEM) {
                    // one TMEM row of BN/2 columns: keys 2c and 2c+1 in column c
                    uint32_t pk[C::BN / 2];
#pragma unroll
                    for (int c2 = 0; c2 < C::BN / 2; ++c2) {
                        const int c = 2 * c2;
                        const float2 x = fma2(make_float2(__uint_as_float(sr[c >> 5][c & 31]),
                                                          __uint_as_float(sr[(c + 1) >> 5][(c + 1) & 31])),
                                              al2, nm2);
                        const float2 p = make_float2(fast_exp2(x.x), fast_exp2(x.y));
                        ps2[c2 & 1] = add2(ps2[c2 & 1], p);
                        pk[c2] = pack_bf16x2(p.x, p.y);
                    }
                    const uint32_t pt = lane_base + C::P_COL + (j % C::NP) * (C::BN / 2);
                    if constexpr (C::BN / 2 == 32) {
                        tmem_st32(pt, pk);
                    } else {
                        tmem_st16(pt, pk);
                    }
                    tmem_wait_st();
                } else {
                    uint8_t *prow = prow_base + (j % C::NP) * C::P_BYTES;
#pragma unroll
                    for (int u = 0; u < C::BN / 8; ++u) {
                        uint32_t w[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int c = u * 8 + e * 2;
                            const float2 x = fma2(make_float2(__uint_as_float(sr[c >> 5][c & 31]),
                                                              __uint_as_float(sr[(c + 1) >> 5][(c + 1) & 31])),
                                                  al2, nm2);
                            const float2 p = make_float2(fast_exp2(x.x), fast_exp2(x.y));
                            ps2[e & 1] = add2(ps2[e & 1], p);
                            w[e] = pack_bf16x2(p.x, p.y);
                        }
                        *reinterpret_cast<uint4 *>(prow + ((u ^ (lr & 7)) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
                    }
                    fence_proxy_async_shared();
                }
                l += (ps2[0].x + ps2[1].x) + (ps2[0].y + ps2[1].y);
                tc_fence_before_sync();
            }
            mbar_arrive(&p_ready[sb]);
        }

        if (failed) {
            flag_error(a.err, kErrTimeout);
            *abort_flag = 1;
        }
        pdl_launch_dependents();
        bool have_o = false;
        if (!failed && n_it > 0) {
            // All MMAs done: `fin` completes once, after the issuer's last PV.  (Waiting
            // on o_done's parity here would be ambiguous: when QK(j+1) is issued
            // before PV(j), the row threads can reach this point two PV phases
            // ahead of o_done, and a parity wait cannot tell phase n-1 from n-3.)
            const bool od = mbar_wait_bounded(fin, 0, a.wait_limit_ns, abort_flag) && !*abort_flag;
            have_o = __all_sync(0xffffffffu, od);
            if (!have_o) {
                flag_error(a.err, kErrTimeout);
                *abort_flag = 1;
            }
        }
        if (have_o && !idle) {
            tc_fence_after_sync();
            const float inv = l > 0.f ? 1.f / l : 0.f;
            const float lse2 = l > 0.f ? m_ref + log2f(l) : -INFINITY;
            const bool real = r < a.Mq;
            const int h = g * a.G + (r % a.G);
            const int unit = b * a.Hkv + g;
            __nv_bfloat16 *dst = a.out + ((size_t(b) * a.Sq + i_row) * a.Hq + h) * D;
            const size_t prow_i = (size_t(unit) * a.Mq + r) * a.num_splits + split;
            float *pdst = a.o_part + prow_i * D;
#pragma unroll 1
            for (int c = 0; c < D / 32; ++c) {
                uint32_t ov[32];
                tmem_ld32(lane_base + C::O_COL + c * 32, ov);
                tmem_wait_ld();
                if (!real) continue;
                if (a.num_splits == 1) {
                    uint32_t pk[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        pk[e] = pack_bf16x2(__uint_as_float(ov[2 * e]) * inv, __uint_as_float(ov[2 * e + 1]) * inv);
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        *reinterpret_cast<uint4 *>(dst + c * 32 + e * 8) =
                            make_uint4(pk[4 * e], pk[4 * e + 1], pk[4 * e + 2], pk[4 * e + 3]);
                } else {
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        *reinterpret_cast<float4 *>(pdst + c * 32 + e * 4) =
                            make_float4(__uint_as_float(ov[4 * e]) * inv, __uint_as_float(ov[4 * e + 1]) * inv,
                                        __uint_as_float(ov[4 * e + 2]) * inv, __uint_as_float(ov[4 * e + 3]) * inv);
                }
            }
            if (real) {
                if (a.num_splits == 1) {
                    if (a.lse != nullptr) a.lse[(size_t(b) * a.Hq + h) * a.Sq + i_row] = lse2 * 0.69314718055994530942f;
                } else {
                    a.lse_part[prow_i] = lse2;
                }
            }
        }
    }

    // ---- teardown (issuer and softmax warps): every TMEM access and MMA is done; free TMEM
    tc_fence_before_sync();
    asm volatile("bar.sync 2, 160;" ::: "memory");
    if (warp == C::ISSUER) {
        tc_fence_after_sync();
        tmem_dealloc(tbase, C::TMEM_COLS);
    }
}

}  // namespace gqa
