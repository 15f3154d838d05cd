// gqa_paged_kernel.cuh -- sparse paged GQA decode with an FP8 E4M3FN K/V pool
// and a sigmoid output gate (sm_103a).
//
// The operation is the one of "Sparse paged GQA decode attention with FP8 KV
// cache on SM89", sections "Workload" and "Implementations": per request, a
// list of top-K logical token indices is mapped through the request's page
// table (page = table[t / page_size], slot = t % page_size) to rows of a
// shared FP8 pool; attention runs over those rows only, with k_scale folded
// into the score multiplier together with the softmax scale and log2(e)
// (base-2 exponentials), v_scale applied once to the output, then
// out = sigmoid(gate) * attn.
//
// Mapping: one CTA per (request, block of up to 8 KV heads); one warp per KV
// head owning that head's whole group of G = Hq / Hkv query heads.  Unlike the
// page's per-warp design, the warp loads each selected K/V row exactly once for
// the whole group (the page's open problem: its grouped kernels fetched each
// row once per query head).  Rows are gathered straight into registers in the
// layout of the tensor-core fragments: K rows as B operands of S = Q K^T (the
// head dimension is permuted consistently in Q and K, which a dot product
// allows), V rows byte-interleaved across token pairs as B operands of
// O = P V.  FP8 codes are widened to f16 with the packed cvt instruction --
// exact, since every E4M3FN value is an f16 value -- and the MMAs run in f16
// with fp32 accumulation.  q is converted to f16 per row with a power-of-two
// row scale (folded back into the score multiplier), so no q value overflows.
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

__device__ __forceinline__ uint4 ldg_stream16(const void *p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

__device__ __forceinline__ uint2 ldg_stream8(const void *p) {
    uint2 r;
    asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0, %1}, [%2];" : "=r"(r.x), "=r"(r.y) : "l"(p));
    return r;
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t r;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
    return r;
}

template <int D>
struct PagedCfg {
    static_assert(D == 64 || D == 128, "paged kernel supports D = 64 or 128");
    static constexpr int KU = D / 64;       // 16-byte K pieces per lane per token (lane owns D/4 bytes)
    static constexpr int KSTEPS = D / 16;   // MMA k-steps over the head dimension
    static constexpr int VB = D / 8;        // V bytes per lane per token
    static constexpr int DT = D / 8;        // output d-tiles of 8
};

// Lane (n = lane/4, c = lane%4) holds, for k-step kk, head-dimension bytes
// d0(kk) .. d0(kk)+3 of its K rows, where d0 = (kk/4) * 64 + 16c + 4 (kk%4).
__device__ __forceinline__ int k_dbase(int kk, int c) { return (kk >> 2) * 64 + 16 * c + 4 * (kk & 3); }

template <int D>
__global__ void __launch_bounds__(32 * kPagedHeadsPerCta, 2) gqa_paged_fp8_kernel(const PagedArgs a) {
    using C = PagedCfg<D>;
    __shared__ int rows_s[kPagedChunk];
    // Q fragments, per warp / k-step / lane (registers are the scarce resource here)
    __shared__ uint4 qf_s[kPagedHeadsPerCta][C::KSTEPS][32];

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int b = blockIdx.y;
    const int g = blockIdx.x * kPagedHeadsPerCta + warp;
    const bool active = g < a.Hkv;
    const int n = lane >> 2;
    const int c = lane & 3;

    // ---- Q fragments (f16, per-row power-of-two scale), staged in shared memory
    float alpha_r[2];
    {
    uint32_t qf[C::KSTEPS][4];
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
        const int hl = n + 8 * hr;
        const bool real = active && hl < a.G;
        float qv[C::KSTEPS][4];
        float mx = 0.f;
#pragma unroll
        for (int kk = 0; kk < C::KSTEPS; ++kk) {
            if (real) {
                const __nv_bfloat16 *src = a.q + (size_t(b) * a.Hq + g * a.G + hl) * D + k_dbase(kk, c);
                const uint2 raw = *reinterpret_cast<const uint2 *>(src);
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
        // 2^e with mx * 2^-e < 2^15: no overflow in f16 (max 65504).
        int ex = 0;
        if (mx >= 32768.f) ex = ilogbf(mx) - 14;
        const float down = ldexpf(1.f, -ex);
        alpha_r[hr] = a.alpha * ldexpf(1.f, ex);
#pragma unroll
        for (int kk = 0; kk < C::KSTEPS; ++kk) {
            qf[kk][hr] = pack_f16x2(qv[kk][0] * down, qv[kk][1] * down);      // k = 2c, 2c+1
            qf[kk][2 + hr] = pack_f16x2(qv[kk][2] * down, qv[kk][3] * down);  // k = 2c+8, 2c+9
        }
    }
#pragma unroll
    for (int kk = 0; kk < C::KSTEPS; ++kk) qf_s[warp][kk][lane] = make_uint4(qf[kk][0], qf[kk][1], qf[kk][2], qf[kk][3]);
    }
    __syncwarp();

    float m_run[2] = {-INFINITY, -INFINITY};
    float l_run[2] = {0.f, 0.f};
    float o[C::DT][4];
#pragma unroll
    for (int nt = 0; nt < C::DT; ++nt) o[nt][0] = o[nt][1] = o[nt][2] = o[nt][3] = 0.f;

    const size_t head_off = size_t(active ? g : 0) * D;
    const size_t row_stride = size_t(a.Hkv) * D;
    bool bad = false;

    for (int base = 0; base < a.topk_n; base += kPagedChunk) {
        const int cn = min(kPagedChunk, a.topk_n - base);
        __syncthreads();  // previous chunk fully consumed
        for (int k = threadIdx.x; k < cn; k += blockDim.x) {
            const int t = __ldg(a.topk + size_t(b) * a.topk_n + base + k);
            rows_s[k] = paged_token_row(a.page_table, b, a.pages_per_req, a.page_size, a.num_pages, t, &bad);
        }
        __syncthreads();
        if (!active) continue;

        for (int s0 = 0; s0 < cn; s0 += 16) {
            // ---- gather K rows (tokens n and n+8 of this step) and V rows
            // (tokens 2c, 2c+1, 2c+8, 2c+9) straight into registers
            int krow[2], vrow[4];
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int k = s0 + n + 8 * j;
                krow[j] = k < cn ? rows_s[k] : -1;
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int k = s0 + 2 * c + (j & 1) + 8 * (j >> 1);
                vrow[j] = k < cn ? rows_s[k] : -1;
            }
            uint4 kr[2][C::KU];
#pragma unroll
            for (int j = 0; j < 2; ++j)
#pragma unroll
                for (int u = 0; u < C::KU; ++u) {
                    if (krow[j] >= 0)
                        kr[j][u] = ldg_stream16(a.k_pool + size_t(krow[j]) * row_stride + head_off + u * 64 + 16 * c);
                    else
                        kr[j][u] = make_uint4(0, 0, 0, 0);
                }
            uint32_t vr[4][C::VB / 4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                if constexpr (C::VB == 16) {
                    uint4 x = make_uint4(0, 0, 0, 0);
                    if (vrow[j] >= 0) x = ldg_stream16(a.v_pool + size_t(vrow[j]) * row_stride + head_off + C::VB * n);
                    vr[j][0] = x.x;
                    vr[j][1] = x.y;
                    vr[j][2] = x.z;
                    vr[j][3] = x.w;
                } else {
                    uint2 x = make_uint2(0, 0);
                    if (vrow[j] >= 0) x = ldg_stream8(a.v_pool + size_t(vrow[j]) * row_stride + head_off + C::VB * n);
                    vr[j][0] = x.x;
                    vr[j][1] = x.y;
                }
            }

            // ---- S = Q K^T  (16 query rows x 16 tokens)
            float s[2][4];
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
#pragma unroll
            for (int kk = 0; kk < C::KSTEPS; ++kk) {
                const uint4 qv4 = qf_s[warp][kk][lane];
                const uint32_t qa[4] = {qv4.x, qv4.y, qv4.z, qv4.w};
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) {
                    const uint4 &x = kr[nt][kk >> 2];
                    const uint32_t w = (kk & 3) == 0 ? x.x : (kk & 3) == 1 ? x.y : (kk & 3) == 2 ? x.z : x.w;
                    const uint32_t b0 = e4m3x2_to_f16x2(uint16_t(w & 0xffffu));
                    const uint32_t b1 = e4m3x2_to_f16x2(uint16_t(w >> 16));
                    mma_f16_16816(s[nt], qa, b0, b1);
                }
            }

            // ---- mask padding, online softmax (base 2)
            float corr[2];
#pragma unroll
            for (int hr = 0; hr < 2; ++hr) {
                float mx = -INFINITY;
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int k = s0 + nt * 8 + 2 * c + e;
                        const bool valid = k < cn && rows_s[k] >= 0;
                        float t = valid ? s[nt][2 * hr + e] * alpha_r[hr] : -INFINITY;
                        s[nt][2 * hr + e] = t;
                        mx = fmaxf(mx, t);
                    }
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
                const float m_new = fmaxf(m_run[hr], mx);
                const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
                corr[hr] = fast_exp2(m_run[hr] - m_use);
                m_run[hr] = m_new;
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                    for (int e = 0; e < 2; ++e) s[nt][2 * hr + e] = fast_exp2(s[nt][2 * hr + e] - m_use);
            }
            // P in f16 as the A operand; the normaliser sums the fp32 weights.
            uint32_t pf[4];
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                pf[nt * 2 + 0] = pack_f16x2(s[nt][0], s[nt][1]);
                pf[nt * 2 + 1] = pack_f16x2(s[nt][2], s[nt][3]);
            }
#pragma unroll
            for (int hr = 0; hr < 2; ++hr)
                l_run[hr] = l_run[hr] * corr[hr] + (s[0][2 * hr] + s[0][2 * hr + 1] + s[1][2 * hr] + s[1][2 * hr + 1]);
#pragma unroll
            for (int nt = 0; nt < C::DT; ++nt) {
                o[nt][0] *= corr[0];
                o[nt][1] *= corr[0];
                o[nt][2] *= corr[1];
                o[nt][3] *= corr[1];
            }

            // ---- O += P V.  B fragment of d-tile t: b0 = (tok 2c, tok 2c+1),
            // b1 = (tok 2c+8, tok 2c+9) at head-dim byte n * VB + t.
#pragma unroll
            for (int w = 0; w < C::VB / 4; ++w) {
                const uint32_t ab01 = prmt(vr[0][w], vr[1][w], 0x5140u);  // bytes 0,1 of tok 2c / 2c+1
                const uint32_t ab23 = prmt(vr[0][w], vr[1][w], 0x7362u);  // bytes 2,3
                const uint32_t cd01 = prmt(vr[2][w], vr[3][w], 0x5140u);
                const uint32_t cd23 = prmt(vr[2][w], vr[3][w], 0x7362u);
                mma_f16_16816(o[4 * w + 0], pf, e4m3x2_to_f16x2(uint16_t(ab01 & 0xffffu)),
                              e4m3x2_to_f16x2(uint16_t(cd01 & 0xffffu)));
                mma_f16_16816(o[4 * w + 1], pf, e4m3x2_to_f16x2(uint16_t(ab01 >> 16)),
                              e4m3x2_to_f16x2(uint16_t(cd01 >> 16)));
                mma_f16_16816(o[4 * w + 2], pf, e4m3x2_to_f16x2(uint16_t(ab23 & 0xffffu)),
                              e4m3x2_to_f16x2(uint16_t(cd23 & 0xffffu)));
                mma_f16_16816(o[4 * w + 3], pf, e4m3x2_to_f16x2(uint16_t(ab23 >> 16)),
                              e4m3x2_to_f16x2(uint16_t(cd23 >> 16)));
            }
        }
    }
    if (bad) flag_error(a.err, kErrIndex);
    if (!active) return;

    // ---- epilogue: v_scale, normalise, sigmoid gate, bf16
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
        l_run[hr] += __shfl_xor_sync(0xffffffffu, l_run[hr], 1);
        l_run[hr] += __shfl_xor_sync(0xffffffffu, l_run[hr], 2);
    }
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
        const int hl = n + 8 * hr;
        if (hl >= a.G) continue;
        const int h = g * a.G + hl;
        const float L = l_run[hr];
        const float f = L > 0.f ? a.v_scale / L : 0.f;
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            // d = (2c + e) * DT + t for d-tiles t = 0 .. DT-1: one contiguous run
            const int d0 = (2 * c + e) * C::DT;
            const size_t off = (size_t(b) * a.Hq + h) * D + d0;
            uint32_t packed[C::DT / 2];
#pragma unroll
            for (int t = 0; t < C::DT; t += 2) {
                const uint32_t graw = *reinterpret_cast<const uint32_t *>(a.gate + off + t);
                const float g0 = __uint_as_float(graw << 16);
                const float g1 = __uint_as_float(graw & 0xffff0000u);
                const float s0 = 1.f / (1.f + __expf(-g0));
                const float s1 = 1.f / (1.f + __expf(-g1));
                packed[t / 2] = pack_bf16x2(o[t][2 * hr + e] * f * s0, o[t + 1][2 * hr + e] * f * s1);
            }
#pragma unroll
            for (int t = 0; t < C::DT / 2; t += 4)
                *reinterpret_cast<uint4 *>(a.out + off + 2 * t) =
                    make_uint4(packed[t], packed[t + 1], packed[t + 2], packed[t + 3]);
        }
        if (a.lse != nullptr && c == 0)
            a.lse[size_t(b) * a.Hq + h] = L > 0.f ? (m_run[hr] + log2f(L)) * 0.69314718055994530942f : -INFINITY;
    }
}

// Test hook: byte copy of the selected rows through the kernel's own index map.
__global__ void gqa_paged_gather_kernel(const uint8_t *pool, const int32_t *page_table, const int32_t *topk,
                                        uint8_t *out, int Hkv, int D, int page_size, int pages_per_req,
                                        int num_pages, int topk_n, unsigned *err) {
    const int k = blockIdx.x;
    const int b = blockIdx.y;
    bool bad = false;
    const int t = topk[size_t(b) * topk_n + k];
    const int row = paged_token_row(page_table, b, pages_per_req, page_size, num_pages, t, &bad);
    if (bad && threadIdx.x == 0) flag_error(err, kErrIndex);
    const int n16 = Hkv * D / 16;
    uint4 *dst = reinterpret_cast<uint4 *>(out + (size_t(b) * topk_n + k) * Hkv * D);
    for (int u = threadIdx.x; u < n16; u += blockDim.x) {
        uint4 v = make_uint4(0, 0, 0, 0);
        if (row >= 0) v = *reinterpret_cast<const uint4 *>(pool + size_t(row) * Hkv * D + size_t(u) * 16);
        dst[u] = v;
    }
}

// Test hook: the kernel's E4M3FN -> f16 widening, reported as fp32.
__global__ void gqa_fp8_to_f32_kernel(const uint8_t *codes, float *out, int n) {
    const int i = (blockIdx.x * blockDim.x + threadIdx.x) * 2;
    if (i >= n) return;
    const uint16_t two = uint16_t(codes[i]) | (i + 1 < n ? uint16_t(codes[i + 1]) << 8 : uint16_t(0));
    const uint32_t h2 = e4m3x2_to_f16x2(two);
    const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&h2));
    out[i] = f.x;
    if (i + 1 < n) out[i + 1] = f.y;
}

}  // namespace gqa
