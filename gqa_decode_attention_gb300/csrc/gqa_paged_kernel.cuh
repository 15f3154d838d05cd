// gqa_paged_kernel.cuh -- paged GQA decode over a shared K/V pool (sm_103a):
// the sparse top-K form with an FP8 E4M3FN pool and a sigmoid output gate,
// and the whole-request form (every token of each request up to its own
// length) over a bf16, FP8 or int8 pool.
//
// The sparse operation is the one of "Sparse paged GQA decode attention with
// FP8 KV cache on SM89", sections "Workload" and "Implementations": per
// request, a list of top-K logical token indices is mapped through the
// request's page table (page = table[t / page_size], slot = t % page_size) to
// rows of a shared FP8 pool; attention runs over those rows only, with
// k_scale folded into the score multiplier together with the softmax scale
// and log2(e) (base-2 exponentials), v_scale applied once to the output, then
// out = sigmoid(gate) * attn.  The whole-request form walks tokens
// 0 .. seq_len-1 of each request through the same page table (the serving
// layout the pages leave open) and masks query row i of S_q to tokens
// t <= seq_len - S_q + i.  int8 pools hold symmetric codes (value = code *
// scale), the int8 KV cache that "Profiling down to the register, then an
// extension that broke my assumptions twice" leaves open.
//
// Schedule: a CTA serves a block of HB KV heads and one worker's share of the
// 16-token steps of all requests, taken in request order (the balanced
// schedule: every worker gets the same number of steps whatever the length
// mix).  A request that lies inside one worker is written whole; one shared
// by several workers leaves fp32 partials (O / l, log2-domain LSE) that
// gqa_paged_combine_kernel merges.
//
// Mapping: one consumer warp per KV head; each consumer owns its head's whole
// group of G * S_q query rows (at most 16), so every K/V row is fetched from
// HBM once for the group (the page's "Open problem": its grouped kernels
// requested every row once per query head).  A producer warp gathers the
// tokens: per token one bulk asynchronous copy of the block's contiguous K
// piece (HB heads x D elements) and one of its V piece, into a ring of
// shared-memory stages of 16 tokens completed on mbarriers.  The copy engine
// moves whole row pieces, and the ring's rows are padded so every fragment
// read below is free of bank conflicts.
//
// Per 16 tokens a consumer computes, on the tensor cores with fp32
// accumulation (f16 inputs for 8-bit pools, bf16 for bf16 pools),
//   S^T[16 tokens x 8 rows] = K[16 x D] . Q^T[D x 8]     (D/16 MMAs)
//   O^T[D x 8 rows]        += V^T[D x 16] . P^T[16 x 8]  (D/16 MMAs)
// with the query rows in the MMA's N dimension (8 rows per n-tile), so no
// accumulator lane is spent on padding rows of the group.  The head
// dimension is permuted identically in Q and K (a dot product allows it) and
// the output dimension is mapped back in the epilogue, which lets every lane
// read whole 16-byte pieces of its K / V rows.  FP8 codes are widened to f16
// with the packed cvt instruction -- exact, since every E4M3FN value is an
// f16 value; an int8 code c becomes the f16 value c + 1152 by one logic op
// (after a byte permute where needed), exactly; the 1152 is folded into the
// scores for K and taken off O once per row for V.  q is converted to f16 per row with a
// power-of-two row scale folded back into the score multiplier, so no q
// value overflows.
#pragma once

#include "gqa_common.cuh"
#include "gqa_params.h"

namespace gqa {

// Physical pool row (page * page_size + slot) of logical token t of request b,
// or -1 for padding (t < 0).  Out-of-range entries give -1 and set *bad.
__device__ __forceinline__ int paged_token_row(const int32_t *page_table, int b, int pages_per_req, int page_size,
                                               int num_pages, int t, bool *bad) {
    if (t < 0) return -1;
    if (t >= pages_per_req * page_size) {
        *bad = true;
        return -1;
    }
    const int p = __ldg(page_table + size_t(b) * pages_per_req + t / page_size);
    if (p < 0 || p >= num_pages) {
        *bad = true;
        return -1;
    }
    return p * page_size + t % page_size;
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t r;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
    return r;
}

// Biased f16x2 of two int8 codes picked from the bytes of (a, b) by the
// permute selector `sel` (result bytes 0 and 2; bytes 1 and 3 are
// overwritten): one lop3 flips each code's sign bit (code + 128 in
// [0, 255]) and sets the f16 exponent of 1024, giving code + 1152 exactly.
// This is the "magic number" integer-to-floating-point conversion (an
// integer written into the low mantissa bits of a float whose exponent makes
// one mantissa unit worth 1, so the float equals a constant plus the integer;
// H. S. Warren, "Hacker's Delight", chapter "Floating-Point"), here with the
// constant 1024 + 128 left in and taken off later by sums, not per element.
__device__ __forceinline__ uint32_t s8pair_biased(uint32_t a, uint32_t b, uint32_t sel) {
    const uint32_t x = prmt(a, b, sel);
    uint32_t r;
    // per bit: c ? b : (a ^ b) with b = 0x64806480, c = 0xFF00FF00
    asm("lop3.b32 %0, %1, %2, %3, 0x9C;" : "=r"(r) : "r"(x), "r"(0x64806480u), "r"(0xFF00FF00u));
    return r;
}
// Biased f16x2 (code + 1152) of bytes 0 and 2 of x, in place: one lop3.
__device__ __forceinline__ uint32_t s8even_biased(uint32_t x) {
    uint32_t r;
    asm("lop3.b32 %0, %1, %2, %3, 0x9C;" : "=r"(r) : "r"(x), "r"(0x64806480u), "r"(0xFF00FF00u));
    return r;
}

// K/V element types of the paged kernel.
enum : int { kKvBf16 = 0, kKvFp8 = 1, kKvInt8 = 2 };

// Two FP8 E4M3FN codes widened to f16x2, exactly (int8 codes take the biased
// path of s8pair_biased instead).
template <int KVT>
__device__ __forceinline__ uint32_t widen8(uint16_t two) {
    static_assert(KVT == kKvFp8, "widen8 serves FP8 pools");
    return e4m3x2_to_f16x2(two);
}

template <int D, int NT, int HB, bool KV8>
struct PagedCfg {
    static_assert(D == 64 || D == 128, "paged kernel supports D = 64 or 128");
    static_assert(HB >= 1 && HB <= kPagedMaxHeadsPerCta, "heads per CTA");
    static constexpr int T = kPagedStageTokens;
    static constexpr int ELEM = KV8 ? 1 : 2;  // bytes per K/V element
    static constexpr int ROWB = D * ELEM;     // bytes of one head's row
    static constexpr int KU = ROWB / 64;      // 16-byte K pieces per lane per token (the lane owns ROWB/4 bytes)
    static constexpr int KSTEPS = D / 16;     // MMA k-steps over the head dimension
    static constexpr int VB = D / 8 * ELEM;   // V bytes per lane per token
    static constexpr int VW = VB / 4;         // V words per lane per token
    static constexpr int DB = D / 16;         // output d-blocks of 16
    static constexpr int PIECE = HB * ROWB;   // bytes of a token row the CTA copies (its heads)
    // Row strides in the ring.  K: rows gi and gi + 1 of a quarter-warp must
    // sit 16 banks apart (stride = 64 mod 128 bytes); V: rows 2c of a
    // quarter-warp must sit 8 banks apart (stride = 16 mod 64 bytes).
    static constexpr int KRS = PIECE + 64;
    static constexpr int VRS = PIECE + 16;
    static constexpr int STAGE_BYTES = T * (KRS + VRS);
    static constexpr int STAGES_FIT = (96 * 1024) / STAGE_BYTES;
    static constexpr int STAGES = STAGES_FIT < 3 ? 3 : (STAGES_FIT > 8 ? 8 : STAGES_FIT);
    static constexpr int WARPS = HB + 1;      // HB consumers, then the producer
    static constexpr int THREADS = 32 * WARPS;
    static constexpr int BAR_OFF = STAGES * STAGE_BYTES;             // full[STAGES], empty[STAGES]
    static constexpr int MASK_OFF = BAR_OFF + 2 * STAGES * 8;        // valid-token mask per stage
    static constexpr int FLAG_OFF = MASK_OFF + STAGES * 4;           // abort flag
    static constexpr int SCHED_OFF = (FLAG_OFF + 4 + 7) / 8 * 8;     // balanced schedule (4 longs)
    static constexpr int ROWS_OFF = (SCHED_OFF + 32 + 15) / 16 * 16; // physical rows of the pass
    static constexpr int SMEM_BYTES = ROWS_OFF + kPagedChunk * 4;
    static constexpr int IPT = (kPagedChunk + THREADS - 1) / THREADS;  // index-map entries per thread
    static constexpr int MIN_BLOCKS_FIT = (220 * 1024) / (SMEM_BYTES + 1024);
    static constexpr int MIN_BLOCKS = MIN_BLOCKS_FIT < 1 ? 1 : (MIN_BLOCKS_FIT > 8 ? 8 : MIN_BLOCKS_FIT);
    static_assert(STAGE_BYTES % 16 == 0 && KRS % 16 == 0 && VRS % 16 == 0, "bulk copy alignment");
};

// Head-dimension element where lane (gi, c) holds, for k-step kk, the four
// elements of its K row that feed the MMA's k = 2c, 2c+1 (first pair) and
// k = 2c+8, 2c+9 (second pair); Q is loaded at the same elements.
//  FP8: word kk%4 of the lane's 16-byte piece kk/4, at byte (kk/4)*64 + 16c.
//  bf16: words 2(kk%2), 2(kk%2)+1 of the lane's piece kk/2, at byte (kk/2)*64 + 16c.
template <bool KV8>
__device__ __forceinline__ int k_dbase(int kk, int c) {
    if constexpr (KV8) return (kk >> 2) * 64 + 16 * c + 4 * (kk & 3);
    return (kk >> 1) * 32 + 8 * c + 4 * (kk & 1);
}

// Head-dimension element of output d-block t, half `hi` (0: accumulator row
// gi, 1: row gi + 8) held by lane gi.
//  FP8: the lane's V piece is bytes VB*gi .. VB*gi + VB-1; block t uses bytes 2t, 2t+1.
//  bf16: the lane's V words are 16-byte chunks at elements 64m + 8gi; block t
//  uses word t, i.e. chunk t/4, elements 2(t%4), 2(t%4)+1.
template <int D, bool KV8>
__device__ __forceinline__ int out_d(int t, int hi, int gi) {
    if constexpr (KV8) return (D / 8) * gi + 2 * t + hi;
    return 64 * (t >> 2) + 8 * gi + 2 * (t & 3) + hi;
}

template <int D, int NT, int HB, int KVT, bool RANGE>
__global__ void __launch_bounds__(PagedCfg<D, NT, HB, KVT != kKvBf16>::THREADS,
                                  PagedCfg<D, NT, HB, KVT != kKvBf16>::MIN_BLOCKS)
    gqa_paged_kernel(const PagedArgs a) {
    constexpr bool KV8 = KVT != kKvBf16;  // 8-bit codes (FP8 or int8) widened to f16; else bf16
    using C = PagedCfg<D, NT, HB, KV8>;
    extern __shared__ __align__(128) uint8_t psmem[];
    uint64_t *full = reinterpret_cast<uint64_t *>(psmem + C::BAR_OFF);
    uint64_t *empty = full + C::STAGES;
    uint32_t *vmask = reinterpret_cast<uint32_t *>(psmem + C::MASK_OFF);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(psmem + C::FLAG_OFF);
    int *rows_s = reinterpret_cast<int *>(psmem + C::ROWS_OFF);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int hb0 = blockIdx.x * HB;
    const int nh = min(HB, a.Hkv - hb0);  // heads of this CTA
    const bool producer = warp == HB;
    const int g = hb0 + warp;
    const bool active = !producer && warp < nh;
    const int gi = lane >> 2;
    const int c = lane & 3;
    const uint32_t ring_addr = smem_u32(psmem);

    if (threadIdx.x == 0) {
        for (int st = 0; st < C::STAGES; ++st) {
            mbar_init(full + st, 1);
            mbar_init(empty + st, nh);
        }
        *abort_flag = 0;
        fence_mbarrier_init();
    }
    __syncthreads();     // barriers and flag initialised before anyone reads them
    pdl_wait_primary();  // inputs may be written by the previous kernel in the stream

    bool bad = false;
    // ---- balanced schedule.  Request b holds len_b tokens (its top-K list,
    // or its own tokens 0 .. seq_len-1), i.e. ceil(len_b / 16) steps; worker
    // w = blockIdx.y of W = num_splits takes global steps
    // [w T / W, (w+1) T / W) of the T steps of all requests, in request
    // order, as segments of consecutive requests.
    int seg_b = 0;   // request of the current segment
    long seg_p = 0;  // its first global step
    long w_begin = 0, w_end = 0;
    if constexpr (!RANGE) {
        // every list has topk_n entries: the schedule in closed form
        const long steps = (a.topk_n + C::T - 1) / C::T;
        const long T = steps * a.B;
        const int W = a.num_splits;
        w_begin = long(blockIdx.y) * T / W;
        w_end = (long(blockIdx.y) + 1) * T / W;
        seg_b = steps > 0 ? int(w_begin / steps) : 0;
        seg_p = long(seg_b) * steps;
    } else {
        long* sched = reinterpret_cast<long *>(psmem + C::SCHED_OFF);
        if (warp == 0) {
            const int W = a.num_splits;
            const int cap = a.pages_per_req * a.page_size;
            long T = 0;
            for (int b0 = 0; b0 < a.B; b0 += 32) {
                const int bb = b0 + lane;
                int len = bb >= a.B ? 0 : RANGE ? __ldg(a.seq_lens + bb) : a.topk_n;
                len = len < 0 ? 0 : (len > cap ? cap : len);
                long st = (len + C::T - 1) / C::T;
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) st += __shfl_xor_sync(0xffffffffu, st, off);
                T += st;
            }
            if (a.step_prefix != nullptr && blockIdx.x == 0 && blockIdx.y == 0) {
                // every request's first global step, for the combine kernel
                long Q = 0;
                for (int b0 = 0; b0 < a.B; b0 += 32) {
                    const int bb = b0 + lane;
                    int len = bb < a.B ? __ldg(a.seq_lens + bb) : 0;
                    len = len < 0 ? 0 : (len > cap ? cap : len);
                    const long st = (len + C::T - 1) / C::T;
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
            // first request whose steps reach past `start`
            long P = 0;
            int first = a.B;
            long first_p = T;
            for (int b0 = 0; b0 < a.B && first == a.B; b0 += 32) {
                const int bb = b0 + lane;
                int len = bb >= a.B ? 0 : RANGE ? __ldg(a.seq_lens + bb) : a.topk_n;
                len = len < 0 ? 0 : (len > cap ? cap : len);
                const long st = (len + C::T - 1) / C::T;
                long incl = st;  // inclusive prefix over the 32 requests of this chunk
#pragma unroll
                for (int off = 1; off < 32; off <<= 1) {
                    const long y = __shfl_up_sync(0xffffffffu, incl, off);
                    if (lane >= off) incl += y;
                }
                // An empty request at step P counts as reaching P + 1: it belongs to
                // the worker whose range holds P (the last worker when P = T).
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
    long seg_t = w_begin;  // global step where the current segment starts

    // this warp's KV head's dequantisation scales: the host scalars, times the
    // device-side per-tensor or per-head values when given
    float alpha_w = a.alpha, vscale_w = a.v_scale;
    if (a.k_scales != nullptr && active) {
        const int si = a.n_scales > 1 ? g : 0;
        alpha_w *= __ldg(a.k_scales + si);
        vscale_w *= __ldg(a.v_scales + si);
    }

    const size_t row_bytes = size_t(a.Hkv) * C::ROWB;
    const uint32_t piece = uint32_t(nh) * C::ROWB;
    bool failed = false;
    int gs0 = 0;     // global step index of the pass's first step (mbarrier phases)
    int issued = 0;  // producer: steps issued so far (all of 0 .. issued-1)

    const bool last_worker = int(blockIdx.y) == a.num_splits - 1;
    while (seg_b < a.B && (seg_t < w_end || (last_worker && seg_t == w_end))) {
    // ---- the current segment: tokens [t_begin, t_begin + n_tok) of request seg_b
    const int b = seg_b;
    int seq_len = RANGE ? __ldg(a.seq_lens + b) : a.topk_n;  // tokens of the request (list length in top-K form)
    {
        const int cap = a.pages_per_req * a.page_size;
        if (seq_len < 0 || seq_len > cap) {
            bad = true;
            seq_len = seq_len < 0 ? 0 : cap;
        }
    }
    const long steps_b = (seq_len + C::T - 1) / C::T;
    const long seg_next = min(w_end, seg_p + steps_b);
    const int t_begin = int(seg_t - seg_p) * C::T;  // first token (list entry) of the segment
    const int n_tok = min(int(seg_next - seg_p) * C::T, seq_len) - t_begin;
    // the segment is the whole request: write the final output; otherwise a
    // partial in slot 0 (the worker's first segment) or 1 (its last)
    const bool complete = seg_t == seg_p && seg_next == seg_p + steps_b;
    const int slot = seg_t == w_begin ? 0 : 1;

    // Index map of tokens [base_k, base_k + cn) of the segment into rows_s,
    // batched so each thread has all its top-K loads and then all its
    // page-table loads in flight together.
    auto index_pass = [&](int base_k, int cn) {
        int tk[C::IPT];
#pragma unroll
        for (int u = 0; u < C::IPT; ++u) {
            const int k = threadIdx.x + u * C::THREADS;
            if constexpr (RANGE)
                tk[u] = k < cn ? t_begin + base_k + k : -1;
            else
                tk[u] = k < cn ? __ldg(a.topk + size_t(b) * a.topk_n + t_begin + base_k + k) : -1;
        }
#pragma unroll
        for (int u = 0; u < C::IPT; ++u) {
            const int k = threadIdx.x + u * C::THREADS;
            const int row = paged_token_row(a.page_table, b, a.pages_per_req, a.page_size, a.num_pages, tk[u], &bad);
            if (k < cn) rows_s[k] = row;
        }
    };
    // The segment's first pass runs before the consumers load Q (the previous
    // segment's closing barrier left rows_s free), so the producer starts its
    // copies while Q is still in flight.
    if (n_tok > 0) index_pass(0, min(kPagedChunk, n_tok));
    __syncthreads();

    // ---- Q^T fragments.  Lane gi holds query row gi (+8 per n-tile) at the
    // elements k_dbase(kk, c) .. +3.  FP8 pools: f16 with a per-row
    // power-of-two scale; bf16 pools: the bf16 values as they are.
    uint32_t qf[NT][C::KSTEPS][2];
    float alpha_s[NT][2];
    float m_run[NT][2], l_run[NT][2];
    float lq[NT][2];  // int8: sum of the f16-rounded weights the P.V product used (its V bias is 1152 x this)
    float o[NT][C::DB][4];
    int kmax[NT][2];  // last visible token of the rows this lane holds in S^T (S_q > 1)
    float kbias[NT][2];  // int8: score offset of the biased K (1152 * sum of the row's q)
    if (!producer) {
        float row_alpha[NT];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const int r = gi + 8 * nt;  // row r = i * G + hl of the unit
            const bool real = active && r < a.Mq;
            const int i = real ? r / a.G : 0;
            const int hl = real ? r % a.G : 0;
            const __nv_bfloat16 *qrow = a.q + ((size_t(b) * a.Sq + i) * a.Hq + g * a.G + hl) * D;
            if constexpr (KV8) {
                float qv[C::KSTEPS][4];
                float mx = 0.f;
#pragma unroll
                for (int kk = 0; kk < C::KSTEPS; ++kk) {
                    if (real) {
                        const uint2 raw = *reinterpret_cast<const uint2 *>(qrow + k_dbase<KV8>(kk, c));
                        qv[kk][0] = __uint_as_float(raw.x << 16);
                        qv[kk][1] = __uint_as_float(raw.x & 0xffff0000u);
                        qv[kk][2] = __uint_as_float(raw.y << 16);
                        qv[kk][3] = __uint_as_float(raw.y & 0xffff0000u);
                    } else {
                        qv[kk][0] = qv[kk][1] = qv[kk][2] = qv[kk][3] = 0.f;
                    }
#pragma unroll
                    for (int e = 0; e < 4; ++e) mx = fmaxf(mx, fabsf(qv[kk][e]));
                }
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
                // 2^e with mx * 2^-e < 2^15: no overflow in f16 (max 65504)
                const int ex = mx >= 32768.f ? ilogbf(mx) - 14 : 0;
                const float down = ldexpf(1.f, -ex);
                row_alpha[nt] = alpha_w * ldexpf(1.f, ex);
#pragma unroll
                for (int kk = 0; kk < C::KSTEPS; ++kk) {
                    if constexpr (KVT == kKvInt8) {
                        // int8 K pairs dims (0, 2) and (1, 3) of each 4-byte word (no byte permute)
                        qf[nt][kk][0] = pack_f16x2(qv[kk][0] * down, qv[kk][2] * down);  // k = 2c, 2c+1
                        qf[nt][kk][1] = pack_f16x2(qv[kk][1] * down, qv[kk][3] * down);  // k = 2c+8, 2c+9
                    } else {
                        qf[nt][kk][0] = pack_f16x2(qv[kk][0] * down, qv[kk][1] * down);  // k = 2c, 2c+1
                        qf[nt][kk][1] = pack_f16x2(qv[kk][2] * down, qv[kk][3] * down);  // k = 2c+8, 2c+9
                    }
                }
            } else {
#pragma unroll
                for (int kk = 0; kk < C::KSTEPS; ++kk) {
                    uint2 raw = make_uint2(0u, 0u);
                    if (real) raw = *reinterpret_cast<const uint2 *>(qrow + k_dbase<KV8>(kk, c));
                    qf[nt][kk][0] = raw.x;  // k = 2c, 2c+1
                    qf[nt][kk][1] = raw.y;  // k = 2c+8, 2c+9
                }
                row_alpha[nt] = alpha_w;
            }
        }
        // int8 pools feed K to the MMA biased by +1152 (no subtraction per
        // element); the scores are corrected by 1152 * sum_d q_d of the row,
        // summed over the same f16 q values the MMA reads.
        float qsum[NT];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            float sacc = 0.f;
            if constexpr (KVT == kKvInt8) {
#pragma unroll
                for (int kk = 0; kk < C::KSTEPS; ++kk)
#pragma unroll
                    for (int j = 0; j < 2; ++j) {
                        const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&qf[nt][kk][j]));
                        sacc += f.x + f.y;
                    }
                sacc += __shfl_xor_sync(0xffffffffu, sacc, 1);
                sacc += __shfl_xor_sync(0xffffffffu, sacc, 2);
            }
            qsum[nt] = sacc;
        }
        // score multipliers and visibility of the rows this lane holds in S^T: 8 nt + 2c + e
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                alpha_s[nt][e] = __shfl_sync(0xffffffffu, row_alpha[nt], 4 * (2 * c + e));
                kbias[nt][e] = 1152.f * __shfl_sync(0xffffffffu, qsum[nt], 4 * (2 * c + e));
                const int r = 8 * nt + 2 * c + e;
                kmax[nt][e] = seq_len - a.Sq + (r < a.Mq ? r / a.G : 0);
            }
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            m_run[nt][0] = m_run[nt][1] = -INFINITY;
            l_run[nt][0] = l_run[nt][1] = 0.f;
            lq[nt][0] = lq[nt][1] = 0.f;
#pragma unroll
            for (int t = 0; t < C::DB; ++t) o[nt][t][0] = o[nt][t][1] = o[nt][t][2] = o[nt][t][3] = 0.f;
        }
    }
    const bool causal = RANGE && a.Sq > 1;

    for (int base_k = 0; base_k < n_tok; base_k += kPagedChunk) {
        const int cn = min(kPagedChunk, n_tok - base_k);
        if (base_k > 0) {  // the first pass was mapped before Q was loaded
            __syncthreads();  // previous pass fully consumed
            if (*abort_flag) break;
            index_pass(base_k, cn);
            __syncthreads();
        }
        const int steps = (cn + C::T - 1) / C::T;

        if (producer) {
            // lanes 0..15 copy the K pieces of the stage's 16 tokens, lanes 16..31 the V pieces
            const int tok = lane & (C::T - 1);
            const bool is_v = lane >= C::T;
            const uint8_t *pool = (is_v ? a.v_pool : a.k_pool) + size_t(hb0) * C::ROWB;
            const uint32_t dst_off = is_v ? uint32_t(C::T * C::KRS + tok * C::VRS) : uint32_t(tok * C::KRS);
            for (int s = 0; s < steps && !failed; ++s) {
                const int gs = gs0 + s;
                const int st = gs % C::STAGES;
                if (gs >= C::STAGES) {
                    bool ok = true;
                    if (lane == 0) ok = mbar_wait_bounded(empty + st, ((gs / C::STAGES) - 1) & 1, a.wait_limit_ns, abort_flag);
                    if (!__shfl_sync(0xffffffffu, ok, 0)) {
                        failed = true;
                        break;
                    }
                }
                const int k = s * C::T + tok;
                const int row = k < cn ? rows_s[k] : -1;
                const unsigned valid = __ballot_sync(0xffffffffu, row >= 0);
                issued = gs + 1;
                if (a.fault_mode == 1 && gs == 0) continue;  // test hook: stage never completes
                if (lane == 0) {
                    vmask[st] = valid & 0xffffu;
                    mbar_arrive_expect_tx(full + st, uint32_t(__popc(valid)) * piece);
                }
                __syncwarp();
                if (row >= 0)
                    bulk_load(ring_addr + uint32_t(st * C::STAGE_BYTES) + dst_off, pool + size_t(row) * row_bytes,
                              piece, full + st);
            }
        } else if (active) {
            const uint32_t kcol = uint32_t(warp * C::ROWB);
            for (int s = 0; s < steps; ++s) {
                const int gs = gs0 + s;
                const int st = gs % C::STAGES;
                const uint32_t okw = mbar_wait_bounded(full + st, (gs / C::STAGES) & 1, a.wait_limit_ns, abort_flag);
                if (!__all_sync(0xffffffffu, okw)) {
                    failed = true;
                    break;
                }
                const uint8_t *kst = psmem + st * C::STAGE_BYTES;
                const uint8_t *vst = kst + C::T * C::KRS;
                const uint32_t mask = vmask[st];
                if constexpr (!RANGE) {  // top-K form: the gate rows are read by the epilogue
                    if (a.gate != nullptr && complete && base_k + (s + 1) * C::T >= n_tok && lane < 2 * NT * 8) {
                        // last step of the request: bring this warp's gate rows into L2 for the epilogue
                        const int r = lane >> 1;
                        if (r < a.Mq) {
                            const int hr = g * a.G + r % a.G;
                            prefetch_l2(a.gate + ((size_t(b) * a.Sq + r / a.G) * a.Hq + hr) * D + (lane & 1) * (D / 2));
                        }
                    }
                }

                // token validity of the two tokens this lane holds in S^T (gi, gi + 8)
                const bool tv0 = (mask >> gi) & 1u, tv1 = (mask >> (gi + 8)) & 1u;
                const int tok0 = t_begin + base_k + s * C::T + gi;  // token index (whole-request form)

                // ---- K words of tokens gi and gi + 8
                uint4 kr[2][C::KU];
#pragma unroll
                for (int j = 0; j < 2; ++j)
#pragma unroll
                    for (int u = 0; u < C::KU; ++u)
                        kr[j][u] = *reinterpret_cast<const uint4 *>(kst + (gi + 8 * j) * C::KRS + kcol + u * 64 + 16 * c);
                // ---- V words of tokens 2c, 2c+1, 2c+8, 2c+9 (rows of padding
                // tokens zeroed: their ring slots hold stale bytes).  Read with
                // the K words, before any arithmetic, so the stage goes back to
                // the producer as early as possible: the stream is bound by the
                // bytes in flight, and a stage held through the step's compute
                // is a stage not loading.
                uint32_t vw[4][C::VW];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int tkn = 2 * c + (j & 1) + 8 * (j >> 1);
                    const bool ok = (mask >> tkn) & 1u;
                    const uint8_t *vrow = vst + tkn * C::VRS + kcol;
                    if constexpr (KV8 && C::VB == 8) {
                        const uint2 x = *reinterpret_cast<const uint2 *>(vrow + 8 * gi);
                        vw[j][0] = ok ? x.x : 0u;
                        vw[j][1] = ok ? x.y : 0u;
                    } else {
                        // 16-byte chunks: FP8 one at byte 16 gi; bf16 one per 64 elements at 128 m + 16 gi
#pragma unroll
                        for (int m = 0; m < C::VW / 4; ++m) {
                            const uint4 x = *reinterpret_cast<const uint4 *>(vrow + 128 * m + 16 * gi);
                            vw[j][4 * m + 0] = ok ? x.x : 0u;
                            vw[j][4 * m + 1] = ok ? x.y : 0u;
                            vw[j][4 * m + 2] = ok ? x.z : 0u;
                            vw[j][4 * m + 3] = ok ? x.w : 0u;
                        }
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(empty + st);  // ring slot free for the producer

                // ---- S^T = K . Q^T
                float st_[NT][4];
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) st_[nt][0] = st_[nt][1] = st_[nt][2] = st_[nt][3] = 0.f;
#pragma unroll
                for (int kk = 0; kk < C::KSTEPS; ++kk) {
                    uint32_t af[4];
                    if constexpr (KV8) {
                        const int u = kk >> 2, w = kk & 3;
                        const uint32_t w0 = w == 0 ? kr[0][u].x : w == 1 ? kr[0][u].y : w == 2 ? kr[0][u].z : kr[0][u].w;
                        const uint32_t w1 = w == 0 ? kr[1][u].x : w == 1 ? kr[1][u].y : w == 2 ? kr[1][u].z : kr[1][u].w;
                        if constexpr (KVT == kKvInt8) {  // biased by +1152, corrected in the scores
                            // pairs (byte 0, byte 2) and (byte 1, byte 3): Q is packed to match
                            af[0] = s8even_biased(w0);
                            af[1] = s8even_biased(w1);
                            af[2] = s8even_biased(w0 >> 8);
                            af[3] = s8even_biased(w1 >> 8);
                        } else {
                            af[0] = widen8<KVT>(uint16_t(w0 & 0xffffu));
                            af[1] = widen8<KVT>(uint16_t(w1 & 0xffffu));
                            af[2] = widen8<KVT>(uint16_t(w0 >> 16));
                            af[3] = widen8<KVT>(uint16_t(w1 >> 16));
                        }
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt) mma_f16_16816(st_[nt], af, qf[nt][kk][0], qf[nt][kk][1]);
                    } else {
                        const int u = kk >> 1;
                        const bool hi = kk & 1;
                        af[0] = hi ? kr[0][u].z : kr[0][u].x;
                        af[1] = hi ? kr[1][u].z : kr[1][u].x;
                        af[2] = hi ? kr[0][u].w : kr[0][u].y;
                        af[3] = hi ? kr[1][u].w : kr[1][u].y;
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt) mma_bf16_16816(st_[nt], af, qf[nt][kk][0], qf[nt][kk][1]);
                    }
                }

                // ---- online softmax over the 16 tokens, rows 8 nt + 2c + e
                uint32_t pb[NT][2];
                float corr[NT][2];
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    float pv[4];
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        bool ok0 = tv0, ok1 = tv1;
                        if (causal) {
                            ok0 = ok0 && tok0 <= kmax[nt][e];
                            ok1 = ok1 && tok0 + 8 <= kmax[nt][e];
                        }
                        const float kb = KVT == kKvInt8 ? kbias[nt][e] : 0.f;
                        const float t0 = ok0 ? (st_[nt][e] - kb) * alpha_s[nt][e] : -INFINITY;
                        const float t1 = ok1 ? (st_[nt][2 + e] - kb) * alpha_s[nt][e] : -INFINITY;
                        float mx = fmaxf(t0, t1);
                        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
                        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
                        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
                        const float m_new = fmaxf(m_run[nt][e], mx);
                        const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
                        corr[nt][e] = fast_exp2(m_run[nt][e] - m_use);
                        m_run[nt][e] = m_new;
                        pv[e] = fast_exp2(t0 - m_use);
                        pv[2 + e] = fast_exp2(t1 - m_use);
                        l_run[nt][e] = l_run[nt][e] * corr[nt][e] + pv[e] + pv[2 + e];
                    }
                    // P^T B fragments: b0 = rows gi at tokens 2c, 2c+1; b1 = tokens 2c+8, 2c+9.
                    const uint32_t pk_lo = KV8 ? pack_f16x2(pv[0], pv[1]) : pack_bf16x2(pv[0], pv[1]);  // token gi
                    const uint32_t pk_hi = KV8 ? pack_f16x2(pv[2], pv[3]) : pack_bf16x2(pv[2], pv[3]);  // token gi + 8
                    if constexpr (KVT == kKvInt8) {  // the rounded weights, rows 2c, 2c+1 (rescaled like l_run)
                        const float2 rlo = __half22float2(*reinterpret_cast<const __half2 *>(&pk_lo));
                        const float2 rhi = __half22float2(*reinterpret_cast<const __half2 *>(&pk_hi));
                        lq[nt][0] = lq[nt][0] * corr[nt][0] + rlo.x + rhi.x;
                        lq[nt][1] = lq[nt][1] * corr[nt][1] + rlo.y + rhi.y;
                    }
                    const int src0 = 4 * (2 * c) + (gi >> 1), src1 = 4 * (2 * c + 1) + (gi >> 1);
                    const uint32_t sel = (gi & 1) ? 0x7632u : 0x5410u;
                    pb[nt][0] = prmt(__shfl_sync(0xffffffffu, pk_lo, src0), __shfl_sync(0xffffffffu, pk_lo, src1), sel);
                    pb[nt][1] = prmt(__shfl_sync(0xffffffffu, pk_hi, src0), __shfl_sync(0xffffffffu, pk_hi, src1), sel);
                }
                bool moved = false;
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) moved |= corr[nt][0] != 1.f || corr[nt][1] != 1.f;
                if (__any_sync(0xffffffffu, moved)) {  // a row's running maximum grew: rescale O
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                        for (int t = 0; t < C::DB; ++t) {
                            o[nt][t][0] *= corr[nt][0];
                            o[nt][t][1] *= corr[nt][1];
                            o[nt][t][2] *= corr[nt][0];
                            o[nt][t][3] *= corr[nt][1];
                        }
                }


                // ---- O^T += V^T . P^T, tokens 2c, 2c+1 (a0, a1) and 2c+8, 2c+9 (a2, a3)
                if constexpr (KV8) {
                    // d-block t: rows m = gi (byte 2t) and gi + 8 (byte 2t + 1) of the lane's piece
#pragma unroll
                    for (int w = 0; w < C::VW; ++w) {
                        uint32_t a_t0[4], a_t1[4];
                        if constexpr (KVT == kKvInt8) {
                            // pair (token 2c, 2c+1) of byte k of word w: permute, lop3; the
                            // +1152 bias stays in and is removed per row in the epilogue
                            a_t0[0] = s8pair_biased(vw[0][w], vw[1][w], 0x4400u);
                            a_t0[1] = s8pair_biased(vw[0][w], vw[1][w], 0x5511u);
                            a_t0[2] = s8pair_biased(vw[2][w], vw[3][w], 0x4400u);
                            a_t0[3] = s8pair_biased(vw[2][w], vw[3][w], 0x5511u);
                            a_t1[0] = s8pair_biased(vw[0][w], vw[1][w], 0x6622u);
                            a_t1[1] = s8pair_biased(vw[0][w], vw[1][w], 0x7733u);
                            a_t1[2] = s8pair_biased(vw[2][w], vw[3][w], 0x6622u);
                            a_t1[3] = s8pair_biased(vw[2][w], vw[3][w], 0x7733u);
                        } else {
                            const uint32_t ab01 = prmt(vw[0][w], vw[1][w], 0x5140u);  // bytes 4w, 4w+1 of tokens 2c / 2c+1
                            const uint32_t ab23 = prmt(vw[0][w], vw[1][w], 0x7362u);  // bytes 4w+2, 4w+3
                            const uint32_t cd01 = prmt(vw[2][w], vw[3][w], 0x5140u);
                            const uint32_t cd23 = prmt(vw[2][w], vw[3][w], 0x7362u);
                            a_t0[0] = widen8<KVT>(uint16_t(ab01 & 0xffffu));
                            a_t0[1] = widen8<KVT>(uint16_t(ab01 >> 16));
                            a_t0[2] = widen8<KVT>(uint16_t(cd01 & 0xffffu));
                            a_t0[3] = widen8<KVT>(uint16_t(cd01 >> 16));
                            a_t1[0] = widen8<KVT>(uint16_t(ab23 & 0xffffu));
                            a_t1[1] = widen8<KVT>(uint16_t(ab23 >> 16));
                            a_t1[2] = widen8<KVT>(uint16_t(cd23 & 0xffffu));
                            a_t1[3] = widen8<KVT>(uint16_t(cd23 >> 16));
                        }
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt) {
                            mma_f16_16816(o[nt][2 * w], a_t0, pb[nt][0], pb[nt][1]);
                            mma_f16_16816(o[nt][2 * w + 1], a_t1, pb[nt][0], pb[nt][1]);
                        }
                    }
                } else {
                    // d-block t = word t: rows m = gi (low half) and gi + 8 (high half)
#pragma unroll
                    for (int t = 0; t < C::DB; ++t) {
                        const uint32_t a_t[4] = {prmt(vw[0][t], vw[1][t], 0x5410u), prmt(vw[0][t], vw[1][t], 0x7632u),
                                                 prmt(vw[2][t], vw[3][t], 0x5410u), prmt(vw[2][t], vw[3][t], 0x7632u)};
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt) mma_bf16_16816(o[nt][t], a_t, pb[nt][0], pb[nt][1]);
                    }
                }
            }
        }
        if (failed && lane == 0) {
            flag_error(a.err, kErrTimeout);
            *abort_flag = 1;
        }
        gs0 += steps;
    }
    // ---- epilogue of the segment.  Lane holds rows r = 8 nt + 2c + e at the
    // head-dim elements out_d(t, 0|1, gi) of o[nt][t][e] / o[nt][t][2 + e].
    //  whole request: out = [sigmoid(gate) *] v_scale * O / l (bf16), LSE (natural log);
    //  shared request: fp32 partial v_scale * O / l and the log2-domain LSE in
    //  the worker's slot, merged by the combine kernel.
    if (active && !failed && !*abort_flag) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                float L = l_run[nt][e];
                L += __shfl_xor_sync(0xffffffffu, L, 4);
                L += __shfl_xor_sync(0xffffffffu, L, 8);
                L += __shfl_xor_sync(0xffffffffu, L, 16);
                if constexpr (KVT == kKvInt8) {  // O^T accumulated (v + 1152) p~: take 1152 sum(p~) off
                    float Lq = lq[nt][e];
                    Lq += __shfl_xor_sync(0xffffffffu, Lq, 4);
                    Lq += __shfl_xor_sync(0xffffffffu, Lq, 8);
                    Lq += __shfl_xor_sync(0xffffffffu, Lq, 16);
#pragma unroll
                    for (int t = 0; t < C::DB; ++t) {
                        o[nt][t][e] -= 1152.f * Lq;
                        o[nt][t][2 + e] -= 1152.f * Lq;
                    }
                }
                const int r = 8 * nt + 2 * c + e;
                if (r >= a.Mq) continue;
                const int i = r / a.G;
                const int h = g * a.G + r % a.G;
                const float f = L > 0.f ? vscale_w / L : 0.f;
                const float lse2 = L > 0.f ? m_run[nt][e] + log2f(L) : -INFINITY;
                if (!complete) {
                    const size_t prow =
                        ((((size_t(blockIdx.x) * a.num_splits + blockIdx.y) * 2 + slot) * HB + warp) * a.Mq) + r;
                    float *dst = a.o_part + prow * D;
#pragma unroll
                    for (int t = 0; t < C::DB; ++t)
                        *reinterpret_cast<float2 *>(dst + out_d<D, KV8>(t, 0, gi)) =
                            make_float2(o[nt][t][e] * f, o[nt][t][2 + e] * f);
                    if (gi == 0) a.lse_part[prow] = lse2;
                    continue;
                }
                const size_t off = ((size_t(b) * a.Sq + i) * a.Hq + h) * D;
                uint32_t graw[C::DB];
#pragma unroll
                for (int t = 0; t < C::DB; ++t)
                    graw[t] = a.gate != nullptr
                                  ? __ldg(reinterpret_cast<const unsigned int *>(a.gate + off + out_d<D, KV8>(t, 0, gi)))
                                  : 0u;
                uint32_t packed[C::DB];
#pragma unroll
                for (int t = 0; t < C::DB; ++t) {
                    float s0 = 1.f, s1 = 1.f;
                    if (a.gate != nullptr) {
                        const float g0 = __uint_as_float(graw[t] << 16);
                        const float g1 = __uint_as_float(graw[t] & 0xffff0000u);
                        s0 = __fdividef(1.f, 1.f + __expf(-g0));
                        s1 = __fdividef(1.f, 1.f + __expf(-g1));
                    }
                    packed[t] = pack_bf16x2(o[nt][t][e] * f * s0, o[nt][t][2 + e] * f * s1);
                }
                // output d-blocks 4q .. 4q+3 are 8 contiguous elements
#pragma unroll
                for (int q4 = 0; q4 < C::DB / 4; ++q4)
                    *reinterpret_cast<uint4 *>(a.out + off + out_d<D, KV8>(4 * q4, 0, gi)) =
                        make_uint4(packed[4 * q4], packed[4 * q4 + 1], packed[4 * q4 + 2], packed[4 * q4 + 3]);
                if (a.lse != nullptr && gi == 0)
                    a.lse[(size_t(b) * a.Hq + h) * a.Sq + i] = lse2 * 0.69314718055994530942f;
            }
    }
    __syncthreads();  // every warp's view of the abort flag is the same below
    if (*abort_flag) break;
    // ---- next segment
    if (seg_next == seg_p + steps_b) {  // request finished: on to the next one
        seg_p = seg_next;
        ++seg_b;
    }
    seg_t = seg_next;
    }  // segment loop

    if (bad) flag_error(a.err, kErrIndex);
    if (producer) {
        // Every copy this CTA issued must land before its shared memory is
        // released; after an abort some may not have been waited for.
        for (int st = 0; st < C::STAGES && st < issued; ++st) {
            const int last = st + ((issued - 1 - st) / C::STAGES) * C::STAGES;  // last step issued into st
            if (a.fault_mode == 1 && last == 0) continue;
            if (lane == 0 && !mbar_wait_bounded(full + st, (last / C::STAGES) & 1, a.wait_limit_ns, nullptr))
                flag_error(a.err, kErrTimeout);
        }
    }
}


// Merge of the partials of requests shared by several workers of the
// balanced schedule.  CTA (b, y) merges rows rr = 8 y + warp of request b
// (rr = g * Mq + r), one warp per row.  Thread 0 works out once per CTA which
// workers hold the request's steps (w_first .. w_last; the request's first step
// P_b and step count come from the closed form of the top-K form or from the
// prefix the main kernel recorded); the CTA returns when one worker holds them
// all (that worker wrote the final output).  The threads stage the workers'
// first steps in shared memory, and each warp loads the partials of up to 8
// workers at a time (one round trip for all of them) before merging them in
// worker order with weights 2^(lse_w - max) (a partial that saw no visible
// token has lse = -inf and weight 0).
constexpr int kPagedMergeRows = 8;       // rows (warps) per CTA
constexpr int kPagedMergeStaged = 1024;  // worker boundaries kept in shared memory
constexpr int kPagedMergeBatch = 8;      // workers' partials in flight per warp

template <int D>
__global__ void __launch_bounds__(32 * kPagedMergeRows) gqa_paged_combine_kernel(const PagedArgs a, int HB) {
    __shared__ long wb[kPagedMergeStaged + 1];  // first global step of workers w_first + j
    __shared__ long info[4];                     // w_first, w_last, P_b, T
    pdl_wait_primary();
    const int b = blockIdx.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long W = a.num_splits;
    if (threadIdx.x == 0) {
        long T, Pb, steps_b;
        if (a.seq_lens == nullptr) {  // top-K form: every list has topk_n entries
            const long steps = (a.topk_n + kPagedStageTokens - 1) / kPagedStageTokens;
            T = steps * a.B;
            Pb = steps * b;
            steps_b = steps;
        } else {  // whole-request form: the main kernel recorded every request's first step
            Pb = a.step_prefix[b];
            steps_b = a.step_prefix[b + 1] - Pb;
            T = a.step_prefix[a.B];
        }
        // worker holding global step s: the largest w with floor(w T / W) <= s
        info[0] = steps_b > 0 ? ((Pb + 1) * W - 1) / T : -1;
        info[1] = steps_b > 0 ? ((Pb + steps_b) * W - 1) / T : -1;
        info[2] = Pb;
        info[3] = T;
    }
    __syncthreads();
    const long w_first = info[0], w_last = info[1], Pb = info[2], T = info[3];
    if (w_first == w_last) return;  // one worker (or an empty request): written by the main kernel
    // floor(x / y) for the schedule's products; 32-bit when they fit
    const bool narrow = (unsigned long long)(T + 1) * (unsigned long long)(W + 1) < (1ull << 32);
    auto qdiv = [narrow](long x, long y) -> long {
        return narrow ? long(unsigned(x) / unsigned(y)) : x / y;
    };
    const long nw = w_last - w_first + 1;
    for (long j = threadIdx.x; j <= nw && j <= kPagedMergeStaged; j += 32 * kPagedMergeRows)
        wb[j] = qdiv((w_first + j) * T, W);
    __syncthreads();
    auto wstart = [&](long w) -> long {
        const long j = w - w_first;
        return j <= kPagedMergeStaged ? wb[j] : qdiv(w * T, W);
    };

    const int rr = blockIdx.y * kPagedMergeRows + warp;
    if (rr >= a.Hkv * a.Mq) return;
    const int g = rr / a.Mq, r = rr - g * a.Mq;
    const int hb = g / HB, lh = g - hb * HB;
    constexpr int V = D / 32;  // values per lane
    float m = -INFINITY, L = 0.f;
    float acc[V];
#pragma unroll
    for (int v = 0; v < V; ++v) acc[v] = 0.f;
    for (long w0 = w_first; w0 <= w_last; w0 += kPagedMergeBatch) {
        float l2[kPagedMergeBatch];
        float x[kPagedMergeBatch][V];
        bool ok[kPagedMergeBatch];
#pragma unroll
        for (int k = 0; k < kPagedMergeBatch; ++k) {
            const long w = w0 + k;
            ok[k] = false;
            l2[k] = -INFINITY;
            if (w > w_last) continue;
            const long ws = wstart(w);
            if (ws == wstart(w + 1)) continue;  // a worker with no steps holds nothing
            ok[k] = true;
            const int slot = (w == w_first && ws < Pb) ? 1 : 0;
            const size_t prow = ((((size_t(hb) * W + w) * 2 + slot) * HB + lh) * a.Mq) + r;
            l2[k] = __ldg(a.lse_part + prow);
            if constexpr (V == 4) {
                const float4 x4 = __ldg(reinterpret_cast<const float4 *>(a.o_part + prow * D) + lane);
                x[k][0] = x4.x;
                x[k][1] = x4.y;
                x[k][2] = x4.z;
                x[k][3] = x4.w;
            } else {
                const float2 x2 = __ldg(reinterpret_cast<const float2 *>(a.o_part + prow * D) + lane);
                x[k][0] = x2.x;
                x[k][1] = x2.y;
            }
        }
#pragma unroll
        for (int k = 0; k < kPagedMergeBatch; ++k) {
            if (!ok[k] || l2[k] == -INFINITY) continue;
            const float mn = fmaxf(m, l2[k]);
            const float sc = fast_exp2(m - mn), wgt = fast_exp2(l2[k] - mn);
#pragma unroll
            for (int v = 0; v < V; ++v) acc[v] = acc[v] * sc + wgt * x[k][v];
            L = L * sc + wgt;
            m = mn;
        }
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;
    const int i = r / a.G;
    const int h = g * a.G + (r - i * a.G);
    const size_t off = ((size_t(b) * a.Sq + i) * a.Hq + h) * D + lane * V;
#pragma unroll
    for (int v = 0; v < V; v += 2) {
        float s0 = 1.f, s1 = 1.f;
        if (a.gate != nullptr) {  // sigmoid gate (top-K form)
            const uint32_t graw = __ldg(reinterpret_cast<const unsigned int *>(a.gate + off + v));
            s0 = __fdividef(1.f, 1.f + __expf(-__uint_as_float(graw << 16)));
            s1 = __fdividef(1.f, 1.f + __expf(-__uint_as_float(graw & 0xffff0000u)));
        }
        *reinterpret_cast<uint32_t *>(a.out + off + v) = pack_bf16x2(acc[v] * inv * s0, acc[v + 1] * inv * s1);
    }
    if (a.lse != nullptr && lane == 0)
        a.lse[(size_t(b) * a.Hq + h) * a.Sq + i] = L > 0.f ? (m + __log2f(L)) * 0.69314718055994530942f : -INFINITY;
}

}  // namespace gqa
