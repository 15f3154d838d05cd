/*
 * gqa_decode.h -- C ABI of the GB300 (sm_103a) grouped-query decode attention
 * library (libgqa_decode.so).
 *
 * The operation (web pages on grouped-query decode attention):
 *  - "When the K/V copy costs more than the attention", section "What I was
 *    looking at": several query heads share one KV head, and query head h
 *    reads KV head h // (Hq / Hkv) in place -- K and V are never copied or
 *    expanded to the query head count.  The same page names the two decode
 *    defects this library is built around: a KV walk that is not split across
 *    CTAs, and a query tile sized for prefill that is nearly empty at decode.
 *  - "Attention Kernel Portability Across GPU Architectures", section
 *    "Decode": a decode step reads the whole KV cache once; its traffic is
 *    2 * B * Hkv * N * D * bytes_per_element.
 *  - "Sparse paged GQA decode attention with FP8 KV cache on SM89", sections
 *    "Workload" and "Implementations": the sparse, paged variant -- top-K
 *    selected token indices per request, a page table, page size 16, an FP8
 *    E4M3FN K/V pool with per-tensor k_scale / v_scale (k_scale folded into the
 *    score scale, v_scale applied once on the output), then a sigmoid gate.
 *  - The same page-table addressing over every token of each request up to
 *    its own length (the serving layout), over bf16, FP8 or int8 pools; int8
 *    is the in-kernel dequantised cache that "Profiling down to the register,
 *    then an extension that broke my assumptions twice" leaves open.
 *  - A score head size different from the value head size (the d192x128
 *    flavour of "When the K/V copy costs more than the attention", section
 *    "Limits, and what I'd do next").
 *
 * Readings where the pages are silent (each also listed in the design notes):
 *  - S_q > 1 uses a bottom-right aligned causal mask: query row i of S_q sees
 *    keys j <= S_kv - S_q + i.
 *  - LSE is the natural log of sum_j exp(scale * q.k_j) over visible keys.
 *  - Tensor layouts (all contiguous, row-major, C order):
 *      q, out         bf16  [B, Sq, Hq, D]
 *      k, v           bf16  [B, Skv, Hkv, D]
 *      lse            fp32  [B, Hq, Sq]
 *      k_pool, v_pool uint8 [num_pages, page_size, Hkv, D]  (E4M3FN codes)
 *      page_table     int32 [B, pages_per_req]
 *      topk_idx       int32 [B, topk]  logical token ids, -1 = padding
 *      q, gate, out (paged) bf16 [B, Hq, D];  lse (paged) fp32 [B, Hq]
 *
 * Conventions for every entry point:
 *  - Pointers named as device pointers must be device-accessible memory owned
 *    by the caller; the library never frees them.  Every bf16 / uint8 tensor
 *    pointer must be 16-byte aligned, fp32 and int32 pointers 4-byte aligned
 *    (GQA_ERR_ALIGNMENT otherwise).
 *  - Calls are asynchronous on `stream` (NULL = the legacy default stream)
 *    and never synchronise, except gqa_device_status and gqa_decode_host.
 *  - The returned status covers host-detectable errors.  On any error status
 *    other than GQA_ERR_CUDA nothing has been launched.
 *  - Device-detected problems (an index out of range in the paged path, a
 *    pipeline wait that exceeded its time limit) set a sticky device error
 *    word that gqa_device_status reads and clears.  After a wait that ran
 *    out, the out and lse of that call are undefined (its kernels stop early
 *    and what they leave unwritten may hold earlier contents).
 *  - The library keeps, per device and for the life of the process, the
 *    device addresses of its own device variables (the error word, the
 *    allocation-free scratch), its memory pool and the kernels' raised
 *    shared-memory limits.  Resetting a device's primary context
 *    (cudaDeviceReset) invalidates them: do not call the library on that
 *    device again in the same process.
 *  - scale <= 0 or NaN selects the default 1 / sqrt(D).
 *  - Hq must be a multiple of Hkv.
 */
#ifndef GQA_DECODE_H
#define GQA_DECODE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
struct CUstream_st;
typedef struct CUstream_st *gqa_stream_t;

typedef enum gqa_status {
    GQA_OK = 0,
    GQA_ERR_INVALID_ARG = 1,    /* bad size, null required pointer, Hq % Hkv != 0, Sq > Skv, ... */
    GQA_ERR_UNSUPPORTED = 2,    /* D not in {64, 128, 256}, or a size beyond the library's limits */
    GQA_ERR_ALIGNMENT = 3,      /* a tensor pointer is not 16-byte aligned */
    GQA_ERR_NO_MEMORY = 4,      /* workspace allocation failed or caller workspace too small */
    GQA_ERR_CUDA = 5,           /* a CUDA runtime/driver call or a launch failed */
    GQA_ERR_DEVICE_TIMEOUT = 6, /* device: a pipeline wait exceeded its time limit */
    GQA_ERR_DEVICE_INDEX = 7    /* device: page id or top-K index out of range (paged path) */
} gqa_status;

/* Human-readable name of a status code (static string, never NULL). */
const char *gqa_status_string(gqa_status s);

/* Library version string (static). */
const char *gqa_version(void);

/* ------------------------------------------------------------------------
 * Dense grouped-query decode attention.
 *
 * For every batch row b, query head h (KV head g = h // (Hq/Hkv)) and query
 * row i < Sq:  s_j = scale * q[b,i,h,:] . k[b,j,g,:]  for visible j,
 *   lse[b,h,i] = ln sum_j exp(s_j),  out[b,i,h,:] = sum_j exp(s_j - lse) v[b,j,g,:].
 * The KV walk is split across CTAs (split count chosen from Skv, B*Hkv and
 * the SM count); each CTA owns one (b, g, split) and the group's
 * (Hq/Hkv)*Sq query rows, up to 128 of them, so each K/V byte is read from
 * HBM once per 128 query rows of a group (once for groups of up to 128
 * rows).  When more than one split is used, an LSE-weighted combine kernel
 * produces out / lse.  Where the automatic choice would split the walk and
 * the (b, g, row group) units fit one wave of SMs (head dims 64, 128 and
 * 192x128, up to 32 query rows per CTA, 64 at head dim 128), key-lane CTAs
 * can take over: CTAs
 * whose warps split their walk among themselves and merge in shared memory.
 * A small cache (at most 256 KiB of K and V per unit) then runs as one such
 * CTA per unit -- one launch, no combine, no workspace (the split-count
 * query reports 1) -- and a longer one as SMs / units such CTAs per unit
 * (one wave; a single one, again without combine or workspace, when that
 * fills most SMs).  An explicit split count is always used as given and
 * never takes key lanes.  Two kernel engines serve the dense calls (see
 * gqa_decode_dense_engine): mma.sync, and tcgen05 for head dim 256 and for
 * head dim 128 from Sq >= 8.
 *
 * q, k, v, out : device, bf16, layouts above.   lse : device fp32 or NULL.
 * Limits: 1 <= Sq <= Skv, B >= 1, Hkv >= 1, Hq % Hkv == 0,
 *         (Hq/Hkv)*Sq <= 4096, Skv < 2^31 / Hkv.
 * D in {64, 128, 256}.  Splits start at multiples of 64 keys.
 * Workspace: fp32 partials, allocated stream-ordered on `stream` from a
 * library-owned memory pool and released stream-ordered after the combine;
 * no allocation happens when a single split is used.
 * ------------------------------------------------------------------------ */
gqa_status gqa_decode(const void *q, const void *k, const void *v, void *out, float *lse,
                      int B, int Sq, int Skv, int Hq, int Hkv, int D, float scale,
                      gqa_stream_t stream);

/* Split count gqa_decode would use for this shape on the current device
 * (>= 1), or a negative gqa_status on invalid arguments. */
int gqa_decode_num_splits(int B, int Sq, int Skv, int Hq, int Hkv, int D);

/* Bytes of workspace gqa_decode_ex needs for `num_splits` (0 = automatic
 * choice); 0 when a single split is used.  Returns 0 on invalid arguments. */
size_t gqa_decode_workspace_bytes(int B, int Sq, int Skv, int Hq, int Hkv, int D, int num_splits);

/* gqa_decode with an explicit split count (0 = automatic; the count is
 * clamped to the number of 64-key blocks and then evened out so that every
 * split but the last covers the same number of blocks) and an optional
 * caller workspace.  When
 * `workspace` is NULL the library allocates stream-ordered as gqa_decode
 * does; otherwise `workspace` must be device memory of at least
 * gqa_decode_workspace_bytes(...) bytes, 256-byte aligned, not used by any
 * other work in flight on another stream.  The same split count always
 * gives bitwise-identical results. */
gqa_status gqa_decode_ex(const void *q, const void *k, const void *v, void *out, float *lse,
                         int B, int Sq, int Skv, int Hq, int Hkv, int D, float scale,
                         int num_splits, void *workspace, size_t workspace_bytes,
                         gqa_stream_t stream);

/* Dense decode whose score head size differs from its value head size.
 * The page "When the K/V copy costs more than the attention", section
 * "Limits, and what I'd do next", lists a d192x128 head flavour beside d64
 * and d128: q and K carry Dqk = 192 dims, V and the output Dv = 128.  The
 * operation is gqa_decode's with the dot product over Dqk dims and the
 * weighted sum over Dv dims:
 *   out[b,i,h,:] = sum_j softmax_j(scale * q[b,i,h,:] . k[b,j,g,:]) v[b,j,g,:]
 * Layouts: q [B, Sq, Hq, Dqk], k [B, Skv, Hkv, Dqk], v [B, Skv, Hkv, Dv],
 * out [B, Sq, Hq, Dv] bf16; lse [B, Hq, Sq] fp32 or NULL.
 * Supported (Dqk, Dv): (192, 128), and Dqk == Dv in {64, 128, 256}, which
 * runs exactly what gqa_decode_ex runs.  Other pairs: GQA_ERR_UNSUPPORTED.
 * scale <= 0 or NaN selects 1 / sqrt(Dqk).  num_splits, workspace and every
 * other limit and convention are gqa_decode_ex's; the workspace holds fp32
 * partials of Dv dims per row. */
gqa_status gqa_decode_dv(const void *q, const void *k, const void *v, void *out, float *lse,
                         int B, int Sq, int Skv, int Hq, int Hkv, int Dqk, int Dv, float scale,
                         int num_splits, void *workspace, size_t workspace_bytes,
                         gqa_stream_t stream);

/* Split count gqa_decode_dv would use (>= 1), or a negative gqa_status. */
int gqa_decode_dv_num_splits(int B, int Sq, int Skv, int Hq, int Hkv, int Dqk, int Dv);

/* Which kernel engine a dense call of this shape runs (gqa_decode,
 * gqa_decode_ex, gqa_decode_noalloc, gqa_decode_host with Dqk == Dv, and
 * gqa_decode_dv): GQA_ENGINE_MMA_SYNC (TMA ring + mma.sync, query rows of the
 * group rounded up to 16 per CTA) or GQA_ENGINE_TCGEN05 (TMA ring + tcgen05
 * with the scores and output in tensor memory, 128 query rows per CTA).  Head
 * dim 256 always runs on tcgen05, head dim 128 on tcgen05 from 8 decode rows
 * per head (Sq >= 8), everything else on mma.sync.  The choice depends on
 * (Sq, Dqk, Dv) only, never on the group size, so native GQA and the same
 * call on K/V expanded per query head share a row's arithmetic.  Host-only:
 * touches no device.  Returns a negative gqa_status on invalid arguments. */
#define GQA_ENGINE_MMA_SYNC 0
#define GQA_ENGINE_TCGEN05 1
int gqa_decode_dense_engine(int B, int Sq, int Skv, int Hq, int Hkv, int Dqk, int Dv);

/* Which kernel engine a paged call of this shape runs: the sparse top-K form
 * (gqa_decode_paged_fp8[_dev_scales]; topk_form != 0, kv_dtype and Sq
 * ignored, Sq = 1) or the whole-request form (gqa_decode_paged[_ex,
 * _dev_scales]; topk_form == 0).  GQA_ENGINE_TCGEN05 (bulk copies of whole
 * token rows, E4M3 products on tcgen05 with scores and output in tensor
 * memory) serves FP8 E4M3FN pools of head dim 128 with Hkv a multiple of 8
 * and at most 4 query rows per KV head (Hq/Hkv * Sq <= 4);
 * GQA_ENGINE_MMA_SYNC (bulk copies + mma.sync) serves every other shape.
 * Both give the same results within the stated tolerances; the tcgen05
 * engine represents the query rows and the softmax weights as sums of two
 * E4M3 values (relative error near 2^-8 per weight; weights below about 2^-20
 * of their row's running maximum are dropped).  Host-only: touches no device.
 * Returns a negative gqa_status on invalid arguments. */
int gqa_decode_paged_engine(int B, int Sq, int Hq, int Hkv, int D, int kv_dtype, int topk_form);

/* Bytes of workspace gqa_decode_dv needs for `num_splits` (0 = automatic);
 * 0 when a single split is used or on invalid arguments. */
size_t gqa_decode_dv_workspace_bytes(int B, int Sq, int Skv, int Hq, int Hkv, int Dqk, int Dv,
                                     int num_splits);

/* Allocation-free dense decode.  The pages have no counterpart to this entry
 * point; it exists for callers that cannot allocate device memory while they
 * decode (a memory budget fixed at start-up, real-time loops where an
 * allocation could block or fail, hosts that hand the library only its input
 * and output tensors).  It runs the same kernels as gqa_decode_ex with the
 * same arguments, but the split partials live in a scratch array compiled
 * into the library (GQA_NOALLOC_SCRATCH_BYTES = 32 MiB, present on every GPU
 * that loads the library until the process exits) instead of a workspace, and
 * the call allocates nothing: no cudaMalloc, no pool, no library allocator.
 *  - The caller still passes q, k, v, out and lse as for gqa_decode.
 *  - A shape whose partials need more than the scratch holds
 *    (gqa_decode_workspace_bytes(...) > gqa_decode_noalloc_scratch_bytes())
 *    is refused with GQA_ERR_NO_MEMORY before anything is launched; fewer
 *    splits (num_splits > 0) need less.
 *  - The first call on each device resolves the scratch's device address
 *    with that device current; make that first call before any stream
 *    capture.
 *  - Every call on a device shares the one scratch array and it keeps the
 *    last call's contents.  Nothing in it needs to start at zero: in a call
 *    that completes without a device error, every partial it reads was
 *    written earlier in the same call (after a wait that ran out, out and lse
 *    are undefined, as for every entry point).  Calls that
 *    may overlap on the GPU (different streams, or devices' work not ordered
 *    by the caller) race on the scratch: serialise them. */
#define GQA_NOALLOC_SCRATCH_BYTES (32u << 20)
gqa_status gqa_decode_noalloc(const void *q, const void *k, const void *v, void *out, float *lse,
                              int B, int Sq, int Skv, int Hq, int Hkv, int D, float scale,
                              int num_splits, gqa_stream_t stream);

/* Size in bytes of the scratch array gqa_decode_noalloc uses. */
size_t gqa_decode_noalloc_scratch_bytes(void);

/* End-to-end form with HOST buffers: copies q, k, v host->device, runs
 * gqa_decode, copies out (and lse when non-NULL) device->host and waits for
 * the stream.  Host buffers should be pinned for full copy bandwidth.  Device
 * buffers are allocated and freed stream-ordered inside the call. */
gqa_status gqa_decode_host(const void *q_host, const void *k_host, const void *v_host,
                           void *out_host, float *lse_host,
                           int B, int Sq, int Skv, int Hq, int Hkv, int D, float scale,
                           gqa_stream_t stream);

/* ------------------------------------------------------------------------
 * Sparse paged GQA decode with an FP8 E4M3FN K/V pool and a sigmoid gate.
 *
 * For request b, query head h (KV head g = h // (Hq/Hkv)) and each selected
 * entry k < topk with t = topk_idx[b,k] >= 0:
 *   page p = page_table[b, t / page_size], slot r = t % page_size,
 *   K^ = e4m3fn(k_pool[p, r, g, :]) * k_scale,  V^ = e4m3fn(v_pool[p, r, g, :]) * v_scale,
 *   s_k = scale * q[b,h,:] . K^.
 * attn = softmax(s) V^;  out[b,h,:] = sigmoid(gate[b,h,:]) * attn;
 * lse[b,h] = ln sum_k exp(s_k) of the ungated scores.  Entries with t < 0
 * are padding and skipped; a row with no valid entry gives out = 0 and
 * lse = -inf.  Entries are used with multiplicity.
 *
 * q, gate, out : device bf16 [B, Hq, D].  lse : device fp32 [B, Hq] or NULL.
 * k_pool, v_pool : device uint8 [num_pages, page_size, Hkv, D].
 * page_table : device int32 [B, pages_per_req].  topk_idx : device int32 [B, topk].
 * k_scale, v_scale : host fp32 scalars (per-tensor dequantisation scales).
 * Limits: D in {64, 128}; Hq / Hkv <= 16; topk <= pages_per_req * page_size;
 *         topk <= 65536; num_pages * page_size < 2^31.
 * Indices are trusted for speed; a t >= pages_per_req * page_size or a page
 * id outside [0, num_pages) is skipped and flags GQA_ERR_DEVICE_INDEX in the
 * device error word.  Small batches (requests filling less than half of the
 * GPU's resident CTA slots) are spread over all slots by splitting lists
 * between CTAs; their fp32 partials live in a workspace allocated
 * stream-ordered from a library-owned pool and are merged (gate included) by
 * a second kernel.  Larger batches use one CTA per request and no workspace.
 * ------------------------------------------------------------------------ */
gqa_status gqa_decode_paged_fp8(const void *q, const void *gate,
                                const uint8_t *k_pool, const uint8_t *v_pool,
                                const int32_t *page_table, const int32_t *topk_idx,
                                float k_scale, float v_scale, void *out, float *lse,
                                int B, int Hq, int Hkv, int D, int page_size, int pages_per_req,
                                int num_pages, int topk, float scale, gqa_stream_t stream);

/* gqa_decode_paged_fp8 with the dequantisation scales in device memory:
 * k_scales and v_scales each point to n_scales fp32 values, n_scales = 1 (per
 * tensor) or Hkv (per KV head: KV head g uses [g]).  The kernel reads them
 * when it starts, so earlier work in the stream may write them.
 * GQA_ERR_INVALID_ARG for null scale pointers or another n_scales;
 * GQA_ERR_ALIGNMENT unless 4-byte aligned.  Everything else as
 * gqa_decode_paged_fp8. */
gqa_status gqa_decode_paged_fp8_dev_scales(const void *q, const void *gate,
                                           const uint8_t *k_pool, const uint8_t *v_pool,
                                           const int32_t *page_table, const int32_t *topk_idx,
                                           const float *k_scales, const float *v_scales, int n_scales,
                                           void *out, float *lse,
                                           int B, int Hq, int Hkv, int D, int page_size,
                                           int pages_per_req, int num_pages, int topk, float scale,
                                           gqa_stream_t stream);

/* ------------------------------------------------------------------------
 * Paged decode over whole requests (no top-K selection), bf16 or FP8 pools.
 *
 * The serving layout of a paged KV cache: request b holds tokens
 * t = 0 .. seq_lens[b]-1, token t stored at page page_table[b, t / page_size],
 * slot t % page_size, of the shared pools (the page-table addressing of
 * "Sparse paged GQA decode attention with FP8 KV cache on SM89", section
 * "Workload", applied to every token instead of a top-K list).  For query row
 * i < Sq of request b and query head h (KV head g = h // (Hq/Hkv)), the
 * visible tokens are t <= seq_lens[b] - Sq + i (bottom-right alignment, as in
 * gqa_decode), and
 *   s_t = scale * q[b,i,h,:] . K^_t,  K^ = k * k_scale,  V^ = v * v_scale,
 *   out[b,i,h,:] = softmax(s) V^,  lse[b,h,i] = ln sum_t exp(s_t).
 * A row that sees no token gives out = 0 and lse = -inf.
 *
 * Schedule: for each block of KV heads, W workers (CTAs) share the
 * T = sum_b ceil(seq_lens[b] / 16) steps of 16 tokens of all requests
 * equally -- worker w takes steps [w T / W, (w+1) T / W) in request order --
 * so the load is balanced whatever the length mix.  A request covered by one
 * worker is written directly; one spread over several workers leaves fp32
 * partials (O / l, log2-domain LSE) that a merge kernel combines with
 * LSE weights.  W defaults to one worker per resident CTA slot.
 *
 * q, out : device bf16 [B, Sq, Hq, D].  lse : device fp32 [B, Hq, Sq] or NULL.
 * k_pool, v_pool : device [num_pages, page_size, Hkv, D] of bf16
 *   (kv_dtype GQA_KV_BF16; k_scale and v_scale are ignored), of E4M3FN codes
 *   (GQA_KV_FP8_E4M3FN) or of two's-complement int8 codes (GQA_KV_INT8, the
 *   int8 KV cache dequantised tile by tile inside the kernel that
 *   "Profiling down to the register, then an extension that broke my
 *   assumptions twice" leaves open: value = code * scale); for 8-bit codes
 *   k_scale, v_scale are finite host fp32 per-tensor scales.
 * page_table : device int32 [B, pages_per_req].  seq_lens : device int32 [B].
 * Limits: D in {64, 128}; (Hq / Hkv) * Sq <= 16; pages_per_req * page_size
 *   and num_pages * page_size < 2^31.  Pointers 16-byte aligned (q, out,
 *   pools), 4-byte aligned (page_table, seq_lens, lse).
 * Device-checked: a seq_lens[b] outside [0, pages_per_req * page_size] is
 *   clamped into it, and a page id outside [0, num_pages) is skipped; both
 *   flag GQA_ERR_DEVICE_INDEX in the device error word.
 * Workspace: gqa_decode_paged allocates the partials stream-ordered from a
 *   library-owned pool; gqa_decode_paged_ex takes num_splits = W, the workers
 *   per head block (0 = automatic), and an optional caller workspace
 *   (256-byte aligned, at least gqa_decode_paged_workspace_bytes; NULL =
 *   library pool).
 * ------------------------------------------------------------------------ */
typedef enum { GQA_KV_BF16 = 0, GQA_KV_FP8_E4M3FN = 1, GQA_KV_INT8 = 2 } gqa_kv_dtype;

gqa_status gqa_decode_paged(const void *q, const void *k_pool, const void *v_pool, int kv_dtype,
                            float k_scale, float v_scale, const int32_t *page_table,
                            const int32_t *seq_lens, void *out, float *lse,
                            int B, int Sq, int Hq, int Hkv, int D, int page_size,
                            int pages_per_req, int num_pages, float scale, gqa_stream_t stream);

gqa_status gqa_decode_paged_ex(const void *q, const void *k_pool, const void *v_pool, int kv_dtype,
                               float k_scale, float v_scale, const int32_t *page_table,
                               const int32_t *seq_lens, void *out, float *lse,
                               int B, int Sq, int Hq, int Hkv, int D, int page_size,
                               int pages_per_req, int num_pages, float scale, int num_splits,
                               void *workspace, size_t workspace_bytes, gqa_stream_t stream);

/* gqa_decode_paged_ex for 8-bit pools (GQA_KV_FP8_E4M3FN, GQA_KV_INT8) with
 * the dequantisation scales in device memory: k_scales and v_scales each
 * point to n_scales fp32 values, n_scales = 1 (per tensor) or Hkv (per KV
 * head: KV head g uses [g]).  The kernel reads them when it starts, so
 * earlier work in the stream may write them.  GQA_ERR_INVALID_ARG for a bf16
 * pool, null scale pointers or another n_scales; GQA_ERR_ALIGNMENT unless
 * 4-byte aligned. */
gqa_status gqa_decode_paged_dev_scales(const void *q, const void *k_pool, const void *v_pool, int kv_dtype,
                                       const float *k_scales, const float *v_scales, int n_scales,
                                       const int32_t *page_table, const int32_t *seq_lens,
                                       void *out, float *lse,
                                       int B, int Sq, int Hq, int Hkv, int D, int page_size,
                                       int pages_per_req, int num_pages, float scale, int num_splits,
                                       void *workspace, size_t workspace_bytes, gqa_stream_t stream);

/* Workers per head block the automatic choice uses for this shape on the
 * current device (negative gqa_status on invalid arguments). */
int gqa_decode_paged_num_splits(int B, int Sq, int Hq, int Hkv, int D, int kv_dtype,
                                int page_size, int pages_per_req);

/* Workspace bytes gqa_decode_paged_ex needs for num_splits (0 = automatic);
 * 0 when no workspace is needed or the arguments are invalid. */
size_t gqa_decode_paged_workspace_bytes(int B, int Sq, int Hq, int Hkv, int D, int kv_dtype,
                                        int page_size, int pages_per_req, int num_splits);

/* ------------------------------------------------------------------------
 * Test hooks.  They run the paged kernel's own index mapping and FP8
 * conversion in isolation so those can be checked bit for bit.
 * ------------------------------------------------------------------------ */

/* out[b, k, g, :] = pool[page_table[b, t/ps], t%ps, g, :] for t = topk_idx[b,k];
 * padding (t < 0) and out-of-range entries give zero bytes (out-of-range also
 * flags GQA_ERR_DEVICE_INDEX).  out: device uint8 [B, topk, Hkv, D]. */
gqa_status gqa_paged_gather_fp8(const uint8_t *pool, const int32_t *page_table,
                                const int32_t *topk_idx, uint8_t *out,
                                int B, int Hkv, int D, int page_size, int pages_per_req,
                                int num_pages, int topk, gqa_stream_t stream);

/* out[i] = value of E4M3FN code codes[i] as fp32, through the same in-register
 * conversion the paged kernel uses.  n >= 0 elements, device pointers. */
gqa_status gqa_fp8_e4m3fn_to_f32(const uint8_t *codes, float *out, int n, gqa_stream_t stream);

/* Waits for `stream`, then reads and clears the device error word:
 * GQA_OK, GQA_ERR_DEVICE_TIMEOUT or GQA_ERR_DEVICE_INDEX (GQA_ERR_CUDA if the
 * wait itself failed). */
gqa_status gqa_device_status(gqa_stream_t stream);

/* Sets the time limit, in nanoseconds, of every pipeline wait in the dense
 * and the paged kernels (default 2e9).  Exceeding it aborts the CTA and flags
 * GQA_ERR_DEVICE_TIMEOUT.  0 restores the default; values below 1e6 (1 ms)
 * are raised to 1e6, so that an aborting CTA's bounded drain outlasts every
 * copy still in flight into its shared memory.  Affects later launches on all
 * streams. */
void gqa_set_wait_limit_ns(uint64_t ns);

#ifdef __cplusplus
}
#endif

#endif /* GQA_DECODE_H */
