/*
 * memra_testing.h - test hooks of the decode library (libmemra.so), not part
 * of the decode ABI in memra.h.  The memra pages have no counterpart: they
 * exist so that a test can drive, on a real GPU, the path that every
 * pipeline wait of the split kernel takes when it runs out, and check the
 * quantizer's division-free quotient against the IEEE one.
 *
 * Every wait of the library's kernels is bounded (about 1 s): past the bound
 * the kernel ORs MEMRA_DEVERR_TIMEOUT into *cache->status, stays until the
 * copies it issued itself have landed (each of those waits bounded too), and
 * returns; it never traps and leaves no copy in flight.
 */
#ifndef MEMRA_TESTING_H
#define MEMRA_TESTING_H

#include <stdint.h>

#include "memra.h"

#ifdef __cplusplus
extern "C" {
#endif

/* memra_decode_attn (same arguments, layout and ownership) with two changes
 * inside its split kernel:
 *   - the waits for pages in the main loop give up after page_wait_ns
 *     nanoseconds (1 .. 1e9) instead of about 1 s;
 *   - the CTA of the first split, first KV head and first sequence declares
 *     16 bytes more than the copies of its first page deliver, so the wait
 *     for that page cannot complete: it runs out, sets MEMRA_DEVERR_TIMEOUT
 *     and that CTA's warp leaves its page loop.
 * The waits for the copies still in flight keep the full limit, so the call
 * takes about one second of GPU time.  The output is then invalid (the status
 * says so); the pools, the workspace and any later call are unaffected.
 * Returns MEMRA_ERR_INVALID_ARG for page_wait_ns outside 1 .. 1e9, otherwise
 * what memra_decode_attn returns for these arguments. */
int memra_testing_decode_attn_short_page(const memra_kv_cache *cache, const void *q, const int32_t *page_table,
                                         int32_t max_pages_per_seq, const int32_t *seq_lens, int32_t max_seq_len,
                                         int32_t batch, int32_t q_len, int32_t n_heads, int32_t n_kv_heads,
                                         int32_t head_dim, float sm_scale, void *workspace, size_t workspace_bytes,
                                         void *out, uint64_t page_wait_ns, void *stream);

/* Adds to *mismatches (device, unsigned 64-bit; the caller zeroes it) the
 * number of (x, s) pairs, x every finite fp16 value and s each of the
 * n_scales float32 scales at `scales` (device, 1 .. 65535 of them, each
 * positive and finite), for which the quantizer's division by a scale
 * (the fp8 and NVFP4 rules round the IEEE float32 quotient x / s, and the
 * quantizer computes it from RN(1 / s) without a division) differs from the
 * IEEE quotient in any bit.  Asynchronous on `stream`.  Returns
 * MEMRA_ERR_INVALID_ARG for null pointers or n_scales outside 1 .. 65535. */
int memra_testing_scale_division_mismatches(const float *scales, int32_t n_scales, unsigned long long *mismatches,
                                            void *stream);

#ifdef __cplusplus
}
#endif

#endif /* MEMRA_TESTING_H */
