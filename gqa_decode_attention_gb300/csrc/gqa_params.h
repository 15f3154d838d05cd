// gqa_params.h -- kernel argument blocks and shape constants shared by the
// kernels and the host front end.
#pragma once

#include <stdint.h>
#include <cuda_bf16.h>

namespace gqa {

// Bits of the sticky device error word.
enum : unsigned {
    kErrTimeout = 1u,  // a pipeline wait exceeded its time limit
    kErrIndex = 2u,    // a page id or top-K index was out of range
};

// Granule of the dense kernel's KV splits: every split starts at a multiple
// of this many keys.
constexpr int kSplitKeys = 64;
// Most KV heads (one consumer warp each) a CTA of the paged kernel serves.
constexpr int kPagedMaxHeadsPerCta = 8;
// Selected tokens per stage of the paged kernel's copy pipeline (one MMA tile).
constexpr int kPagedStageTokens = 16;
// Tokens (top-K entries or request tokens) whose pool rows one index-map pass
// of the paged kernel resolves.
constexpr int kPagedChunk = 2048;

struct DenseArgs {
    const __nv_bfloat16 *q;
    __nv_bfloat16 *out;
    float *lse;
    float *o_part;    // [B*Hkv, Mq, splits, D] fp32 (splits > 1)
    float *lse_part;  // [B*Hkv, Mq, splits] fp32, log2 domain (splits > 1)
    int B, Sq, Skv, Hq, Hkv, G, Mq;
    int n_blocks, blocks_per_split, num_splits, row_groups;  // blocks of kSplitKeys keys
    float alpha;  // scale * log2(e)
    unsigned long long wait_limit_ns;
    int fault_mode;  // test hook: 1 = the producer never loads the first tile
    unsigned *err;   // device error word
};

struct PagedArgs {
    const __nv_bfloat16 *q;     // [B, Sq, Hq, D]
    const __nv_bfloat16 *gate;  // [B, Hq, D] or null (no gate)
    const uint8_t *k_pool;      // [num_pages, page_size, Hkv, D] elements (FP8 codes or bf16)
    const uint8_t *v_pool;
    const int32_t *page_table;  // [B, pages_per_req]
    const int32_t *topk;        // [B, topk_n] (top-K form)
    const int32_t *seq_lens;    // [B] (whole-request form)
    __nv_bfloat16 *out;         // [B, Sq, Hq, D]
    float *lse;                 // [B, Hq, Sq] or null
    float *o_part;              // whole-request form, shared requests: [head block, worker, 2 slots, HB, Mq, D] fp32
    float *lse_part;            // [head block, worker, 2 slots, HB, Mq] fp32, log2 domain
    long long *step_prefix;     // whole-request form, several workers: [B + 1] first global step of each request
    int B, Sq, Hq, Hkv, G, Mq, page_size, pages_per_req, num_pages, topk_n;
    int num_splits;             // whole-request form: workers per head block
    float alpha;    // scale * k_scale * log2(e)
    float v_scale;
    // Device-side scales (null: the host scalars above apply): n_scales = 1
    // per tensor or Hkv per KV head; multiply alpha and v_scale.
    const float *k_scales;
    const float *v_scales;
    int n_scales;
    unsigned long long wait_limit_ns;
    int fault_mode;  // test hook: 1 = the producer never issues the first stage
    unsigned *err;   // device error word
};

}  // namespace gqa
