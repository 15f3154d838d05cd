/*
 * gqa_decode_debug.h -- test-only controls of libgqa_decode.so.
 *
 * Not part of the operation's interface; the pages have no counterpart.  They
 * exist so the test suite can exercise the device-side failure path without
 * faulting a GPU.
 */
#ifndef GQA_DECODE_DEBUG_H
#define GQA_DECODE_DEBUG_H

#include <stddef.h>

#include "gqa_decode.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Fault injection for the bounded pipeline waits of the dense and the paged
 * kernels.
 * mode 0: normal operation (default).
 * mode 1: the producer never issues the loads of each CTA's first KV tile
 *         (dense) or first stage of selected rows (paged), so the consumers'
 *         wait on it runs out after the configured wait limit
 *         (gqa_set_wait_limit_ns); the CTA flags GQA_ERR_DEVICE_TIMEOUT in the
 *         device error word, lets its other loads land, and returns.  Outputs
 *         are then undefined.
 * Affects later gqa_decode / gqa_decode_ex / gqa_decode_paged_fp8 launches on
 * all streams. */
void gqa_debug_set_fault_mode(int mode);

/* Measurement hook.  When both are non-NULL, every later dense or paged
 * decode call records `before` on its stream immediately before launching its
 * main kernel (the split kernel, or the paged kernel) and `after` immediately
 * after it, so a caller can time that kernel alone with
 * cudaEventElapsedTime.  The handles are cudaEvent_t created by the caller;
 * pass NULL, NULL to stop.  Recording between the split and the combine
 * kernel serialises the combine's early launch, so use it only to measure. */
void gqa_debug_set_kernel_events(void *before, void *after);

/* Measurement and test hook: mode 1 runs every later paged call on the
 * mma.sync engine, even where gqa_decode_paged_engine reports tcgen05, so
 * the two engines can be compared on the same shapes; mode 0 (default)
 * chooses by shape.  Affects workspace sizes and worker counts computed
 * afterwards as well; set it only between calls. */
void gqa_debug_set_paged_engine(int mode);

/* Measurement hook: reads `bytes` (a multiple of 16) of device memory at
 * `buf` (16-byte aligned) once with 16-byte loads and XORs every 32-bit word
 * into *sink (device memory, 4-byte aligned; the caller owns both).  The
 * benchmark times it to report a read-only HBM rate beside the copy peak: a
 * decode kernel only reads its K/V, so its traffic matches this stream, not a
 * copy's read + write.  Asynchronous on `stream`; GQA_ERR_INVALID_ARG or
 * GQA_ERR_ALIGNMENT before launching for bad arguments. */
gqa_status gqa_debug_read_stream(const void *buf, size_t bytes, unsigned *sink, gqa_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* GQA_DECODE_DEBUG_H */
