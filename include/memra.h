/*
 * memra.h - C ABI of the GB300 (sm_103a) decode-attention library for a
 * block-quantized, paged KV cache.
 *
 * What the library computes (sources are the memra project pages):
 *   - The KV-cache formats are the knobs named on the "memra-bench" card,
 *     section "drafts/kf4/ - archived experiment": K = q8_0 | fp8,
 *     V = q5_1 | q4_0 | fp8, defaults q8_0 / q5_1; and NVFP4 for K or V, the
 *     NVFP4 KV-cache arm that section records as archived.
 *   - Pages are the request-sized, reusable KV allocation of the memra
 *     README ("Request reuse and admission" item of the serving surface);
 *     several page tables may point at the same page (shared prefix, the
 *     README introduction's 4,860-token shared-prefix serving shape).
 *   - Query lengths: 1 (plain decode) and K+1 (MTP speculative verify,
 *     README "Speculative decoding" item); contexts up to the 262,144 tokens
 *     of the README's "Long context and larger models" item.
 *
 * Per-block rules (32 consecutive elements of one fp16 row along head_dim;
 * rne = round half to even of the exact real value, using the stored fp16 d):
 *   q8_0  d = fp16(max|x|/127),  q = clamp(rne(x/d), -127, 127),   x^ = d*q
 *   q5_1  m = min x, d = fp16((max-min)/31), q = clamp(rne((x-m)/d), 0, 31),
 *                                                                  x^ = d*q + m
 *   q4_0  d = fp16(max|x|/7),    q = clamp(rne(x/d), -8, 7),       x^ = d*q
 *   fp8   OCP e4m3 ("fn"): byte = rne_satfinite(fp32(x) / s), x^ = s*e4m3(byte),
 *         s a float32 per-tensor scale given in memra_kv_cache.
 *   nvfp4 blocks of 16 elements, OCP E2M1 codes, an e4m3 scale byte per block
 *         and the float32 per-tensor scale s, each step one float32 operation:
 *         u = max|x| / (6*s), sb = e4m3_rne_satfinite(u),
 *         c = e2m1_rne_satfinite(x / (e4m3(sb)*s)) (c = 0 when sb = 0),
 *         x^ = s * e4m3(sb) * e2m1(c).
 *   A stored d of 0 gives q = 0.  Inputs must be finite.
 *
 * Attention: query row i of sequence b sits at position seq_lens[b]-q_len+i
 * and sees keys 0..seq_lens[b]-q_len+i (causal among the q_len new tokens);
 * query head h reads KV head h / (n_heads / n_kv_heads).  The output is
 * softmax(q K^T * sm_scale) V^ over the dequantized cache, accumulated in
 * float32, written as fp16.
 *
 * Conventions for every entry point:
 *   - Pointers marked "device" are CUDA device pointers; the caller owns all
 *     memory.  The library never allocates, frees or synchronizes on the
 *     compute entry points; work is enqueued on `stream` (a cudaStream_t,
 *     NULL = legacy default stream).
 *   - Return value: a memra_status.  Argument errors are detected on the host
 *     before anything is enqueued.  Errors that only the GPU can see (a page
 *     id outside the pool, a slot outside the pool, a seq_len larger than
 *     the page table or max_seq_len, a pipeline wait that timed out) never
 *     fault: the kernel skips the offending page / row and ORs a
 *     MEMRA_DEVERR_* bit into *cache->status; memra_read_status reports it.
 *   - All pointers must be 16-byte aligned; tensors are dense row-major.
 *
 * Pool layout (part of the ABI).  Each pool is
 *   [num_pages][n_kv_heads][segment]
 * and one segment holds one page (16 tokens) of one KV head.  D = head_dim,
 * nb = D/32.  For token t (0..15) of the page and element j (0..D-1) of its
 * row, b = j/32, r = j%32:
 *   K q8_0 / fp8 codes (a q8_0 byte holds q + 128, an fp8 byte the e4m3 code):
 *       kc = r/8, e = r%8, tg = t%8, tp = t/8, lane = 4*tg+kc,
 *       byte ((tp*(nb/2) + b/2)*32 + lane)*16 + (b%2)*8 + e
 *   K q8_0 d:  16*D + (t*nb + b)*2                       (fp16, little endian)
 *   V: vg = r/4, h = (r%4)/2, s = r%2, c = (t%8)/2, f = t%2, p = t/8,
 *      lane = 4*vg + c, k = 2*f + p
 *   V q5_1 / q4_0 low nibble (q5_1: q & 15; q4_0: q + 8):
 *       byte ((b/2)*32 + lane)*16 + (b%2)*8 + 4*h + k, bits 4*s .. 4*s+3
 *   V q5_1 bit 4 of q: byte 8*D + (lane*(nb/2) + b/2)*4 + k, bit 4*s + 2*(b%2) + h
 *   V q5_1 d: 10*D + ((c*nb + b)*4 + 2*p + f)*2,  m: 11*D + same offset
 *   V q4_0 d: 8*D + ((c*nb + b)*4 + 2*p + f)*2
 *   V fp8:    byte (b*32 + lane)*16 + 8*h + 2*(2*p + s) + f
 *   NVFP4 (two 4-bit codes per byte, low nibble first; b16 = j/16):
 *     K codes: c = r/8, e = r%8, lane = 4*(t%8) + c, w = 2*b + e/4,
 *       byte ((w/4)*32 + lane)*16 + (w%4)*4 + t/8 + 2*((e%4)/2), bits 4*(e%2) ..
 *     K scale byte: 8*D + t*(D/16) + b16
 *     V codes: r16 = j%16, c = (t%8)/2, lane = 4*(r16%8) + c,
 *       byte ((b16/4)*32 + lane)*16 + (b16%4)*4 + t%2 + 2*(t/8), bits 4*(r16/8) ..
 *     V scale byte: 8*D + (c*(D/16) + b16)*4 + t%2 + 2*(t/8)
 * Segment bytes: K q8_0 17*D, K fp8 16*D, K nvfp4 9*D, V q5_1 12*D,
 * V q4_0 9*D, V fp8 16*D, V nvfp4 9*D.  Every byte of a segment belongs to exactly one token, so
 * appends to different slots never touch the same byte.  The order is the
 * register-fragment order of the decode kernel's tensor-core tiles, so one
 * bulk copy per segment lands the page in shared memory ready to read with
 * conflict-free 16-byte loads.
 */
#ifndef MEMRA_H
#define MEMRA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Return codes of every entry point. */
typedef enum {
    MEMRA_OK = 0,
    MEMRA_ERR_INVALID_ARG = 1,   /* a pointer, size or shape is not valid          */
    MEMRA_ERR_UNSUPPORTED = 2,   /* valid, but outside what this build supports    */
    MEMRA_ERR_WORKSPACE = 3,     /* workspace too small                            */
    MEMRA_ERR_CUDA = 4,          /* a CUDA runtime call or launch failed           */
    MEMRA_ERR_DEVICE = 5         /* memra_read_status: the device flagged an error */
} memra_status;

/* Bits the kernels OR into *memra_kv_cache.status. */
#define MEMRA_DEVERR_BAD_PAGE    1   /* page id outside [0, num_pages): page skipped      */
#define MEMRA_DEVERR_BAD_SLOT    2   /* append slot >= num_pages*16: row skipped          */
#define MEMRA_DEVERR_BAD_SEQ_LEN 4   /* seq_len < q_len, > max_seq_len or > table: clamped */
#define MEMRA_DEVERR_TIMEOUT     8   /* a pipeline wait gave up after ~1 s: result invalid */
#define MEMRA_DEVERR_PREFIX     16   /* cascade: a page table differs from the first sequence's
                                        within the shared prefix: that row used the first's pages */

/* KV block formats (the memra-bench card's KV knobs). */
typedef enum {
    MEMRA_KV_Q8_0 = 0,       /* K only */
    MEMRA_KV_Q5_1 = 1,       /* V only */
    MEMRA_KV_Q4_0 = 2,       /* V only */
    MEMRA_KV_FP8_E4M3 = 3,   /* K or V */
    MEMRA_KV_NVFP4 = 4       /* K or V: the memra-bench card's archived "kf4" NVFP4 arm */
} memra_kv_format;

/* Page size (tokens) and the bounds of the split-K plan.  A sequence of T
 * tokens is cut into splits of C(T) tokens, C(T) = clamp(roundup16(ceil(T /
 * S)), MEMRA_SPLIT_TOKENS, MEMRA_SPLIT_TOKENS_MAX), where S = (SMs of the
 * device) x (CTAs per SM of the kernel configuration) / n_kv_heads, so that one
 * long sequence fills the GPU in one wave.  C depends only on the sequence's
 * own length and the device, never on the rest of the batch: a sequence's
 * result bytes are the same alone or batched.  The floor of 1,280 tokens
 * (measured against 1,024 to 2,048 on batch-1 decode from 8K to 256K tokens,
 * batches of 4 to 64, verify and shared prefixes) keeps the per-split fixed
 * cost small where many sequences fill the GPU, without slowing a single
 * sequence of moderate length. */
#define MEMRA_PAGE_SIZE 16
/* Largest q_len (new tokens per sequence: 1 + draft tokens) and largest GQA
 * group n_heads / n_kv_heads that the decode calls take. */
#define MEMRA_MAX_Q_LEN 16
#define MEMRA_MAX_GROUP 128
#define MEMRA_SPLIT_TOKENS 1280
#define MEMRA_SPLIT_TOKENS_MAX 8192

/* A paged KV cache.  Plain data; the caller owns the pools and status word. */
typedef struct {
    int32_t k_fmt;          /* memra_kv_format: MEMRA_KV_Q8_0, _FP8_E4M3 or _NVFP4           */
    int32_t v_fmt;          /* memra_kv_format: MEMRA_KV_Q5_1, _Q4_0, _FP8_E4M3 or _NVFP4    */
    int32_t page_size;      /* must be MEMRA_PAGE_SIZE                                      */
    int32_t n_kv_heads;     /* >= 1                                                          */
    int32_t head_dim;       /* 128 or 256                                                    */
    int32_t num_pages;      /* pages in each pool, >= 1                                      */
    void *k_pool;           /* device, memra_kv_pool_bytes(k_fmt, 0, ...) bytes              */
    void *v_pool;           /* device, memra_kv_pool_bytes(v_fmt, 1, ...) bytes              */
    float k_scale;          /* fp8 / nvfp4 K: float32 per-tensor scale s (x^ = s*e4m3, or
                               s*e4m3(block scale)*e2m1); else ignored                      */
    float v_scale;          /* fp8 / nvfp4 V: same for V                                     */
    int32_t *status;        /* device int32 the kernels OR MEMRA_DEVERR_* bits into; may be NULL */
} memra_kv_cache;

/* Bytes of one segment (one page of one KV head) of a K (is_v = 0) or V
 * (is_v = 1) pool; 0 if the format / side / head_dim combination is not
 * supported.  Host only, no CUDA call. */
size_t memra_kv_segment_bytes(int32_t fmt, int32_t is_v, int32_t head_dim);

/* Bytes of a whole pool: num_pages * n_kv_heads * segment; 0 if unsupported.
 * Host only, no CUDA call. */
size_t memra_kv_pool_bytes(int32_t fmt, int32_t is_v, int32_t num_pages, int32_t page_size,
                           int32_t n_kv_heads, int32_t head_dim);

/* Quantize-append (the write side of the paged cache; formats as above).
 *   k, v          device fp16 [n_tok][n_kv_heads][head_dim]
 *   slot_mapping  device int32 [n_tok]; slot = page*16 + offset.  A negative
 *                 slot skips the row (padding); a slot >= num_pages*16 skips
 *                 it and sets MEMRA_DEVERR_BAD_SLOT.  Slots must be distinct
 *                 within one call.
 * n_tok == 0 is a no-op.  Results are bit-exact under the rules above. */
int memra_kv_append(const memra_kv_cache *cache, const void *k, const void *v,
                    const int32_t *slot_mapping, int32_t n_tok, void *stream);

/* Workspace bytes memra_decode_attn needs for these sizes (the split-K
 * partials: float32 [batch*q_len*n_heads][memra_num_splits(max_seq_len)][head_dim]
 * plus one float32 log-sum-exp per partial; memra_num_splits(max_seq_len)
 * bounds the split count of any sequence).  Host only. */
size_t memra_decode_attn_workspace_bytes(int32_t batch, int32_t q_len, int32_t n_heads,
                                         int32_t head_dim, int32_t max_seq_len);

/* Decode attention over the paged cache (split-K pass, then the combine).
 *   q            device fp16 [batch][q_len][n_heads][head_dim]
 *   page_table   device int32 [batch][max_pages_per_seq]; entries past
 *                ceil(seq_lens[b]/16) are not read
 *   seq_lens     device int32 [batch]; context of each sequence INCLUDING its
 *                q_len new tokens (append them first with memra_kv_append)
 *   max_seq_len  host upper bound of seq_lens (sizes the split grid)
 *   n_kv_heads, head_dim must equal the cache's; n_heads % n_kv_heads == 0;
 *   q_len <= MEMRA_MAX_Q_LEN, n_heads/n_kv_heads <= MEMRA_MAX_GROUP, batch and
 *   n_kv_heads <= 65535 (else MEMRA_ERR_UNSUPPORTED)
 *   sm_scale     softmax scale (1/sqrt(head_dim) for standard attention)
 *   workspace    device, >= memra_decode_attn_workspace_bytes(...) bytes
 *   out          device fp16 [batch][q_len][n_heads][head_dim]
 * Query row i of sequence b sits at position seq_lens[b] - q_len + i and sees
 * keys 0 .. that position.  Each row's result depends only on its visible
 * keys, its query and the device: a verify row (q_len > 1) has the same
 * bytes as a q_len = 1 call at that position, and a sequence has the same
 * bytes alone or in any batch.
 * batch == 0 is a no-op.  A row with no visible key (a sequence shorter than
 * q_len, flagged MEMRA_DEVERR_BAD_SEQ_LEN, or of length 0) yields zeros. */
int memra_decode_attn(const memra_kv_cache *cache, const void *q, const int32_t *page_table,
                      int32_t max_pages_per_seq, const int32_t *seq_lens, int32_t max_seq_len,
                      int32_t batch, int32_t q_len, int32_t n_heads, int32_t n_kv_heads,
                      int32_t head_dim, float sm_scale, void *workspace, size_t workspace_bytes,
                      void *out, void *stream);

/* The two passes of memra_decode_attn, separately (same arguments and
 * meaning).  memra_decode_attn == partials followed by combine on one
 * stream (the combine is left out when max_seq_len <= MEMRA_SPLIT_TOKENS: every row then
 * fits one split).  Rows that fit one split, and rows with no visible key
 * (zeros), are written to `out` by the partials pass directly; the combine
 * pass merges the others. */
int memra_decode_attn_partials(const memra_kv_cache *cache, const void *q, const int32_t *page_table,
                               int32_t max_pages_per_seq, const int32_t *seq_lens, int32_t max_seq_len,
                               int32_t batch, int32_t q_len, int32_t n_heads, int32_t n_kv_heads,
                               int32_t head_dim, float sm_scale, void *workspace, size_t workspace_bytes,
                               void *out, void *stream);
int memra_decode_attn_combine(const memra_kv_cache *cache, const int32_t *seq_lens, int32_t max_seq_len,
                              int32_t max_pages_per_seq, int32_t batch, int32_t q_len, int32_t n_heads,
                              int32_t head_dim, const void *workspace, size_t workspace_bytes, void *out,
                              void *stream);

/* One decode step in a single split-K pass: quantize-append of the step's new
 * rows fused into the attention that reads them (the write and read sides of
 * the memra README's paged, block-quantized cache, "Speculative decoding" for
 * q_len > 1).  Same results as memra_kv_append of the rows at slots
 * page_table[b][pos/16]*16 + pos%16, pos = seq_lens[b]-q_len .. seq_lens[b]-1,
 * followed by memra_decode_attn; the pool bytes are bit-identical.
 *   k_new, v_new  device fp16 [batch][q_len][n_kv_heads][head_dim], 16-byte
 *                 aligned: the K / V rows of the q_len new tokens, in position
 *                 order
 *   other arguments as memra_decode_attn; max_seq_len >= q_len.
 * Each new row is stored by the CTA whose split holds its position, before
 * that CTA copies the page in, so no other launch is needed.  The pages that
 * receive new rows must belong to one sequence of the batch (a page shared by
 * two sequences, e.g. a shared prefix, is read-only here).  Rows whose page
 * id is out of range are skipped (MEMRA_DEVERR_BAD_PAGE); a sequence shorter
 * than q_len stores only the rows with a position >= 0 and sets
 * MEMRA_DEVERR_BAD_SEQ_LEN. */
int memra_decode_step(const memra_kv_cache *cache, const void *k_new, const void *v_new, const void *q,
                      const int32_t *page_table, int32_t max_pages_per_seq, const int32_t *seq_lens,
                      int32_t max_seq_len, int32_t batch, int32_t q_len, int32_t n_heads, int32_t n_kv_heads,
                      int32_t head_dim, float sm_scale, void *workspace, size_t workspace_bytes, void *out,
                      void *stream);

/* Sliding-window attention over ring page tables (the memra README's opt-in
 * SWA ring in its "Recent fixes" list, which right-sizes the KV of sliding-
 * window layers: only the last pages of a sequence are kept, reused modulo
 * the ring).  Same arguments and results as memra_decode_attn /
 * memra_decode_step, except:
 *   ring_table   device int32 [batch][ring_pages]: position p of sequence b
 *                lives in page ring_table[b][(p / 16) % ring_pages], slot p % 16
 *                (memra_kv_append takes those slots)
 *   ring_pages   >= (window + q_len - 2) / 16 + 2, so that the ring holds every
 *                key any query row sees; else MEMRA_ERR_INVALID_ARG
 *   window       >= 1: the row at position p sees keys max(0, p - window + 1) .. p
 *   seq_lens     are not bounded by the ring (only by max_seq_len)
 * The workspace is memra_decode_attn_workspace_bytes(...) of the same sizes.
 * Verify rows stay byte-identical to q_len = 1 calls at their positions. */
int memra_decode_attn_window(const memra_kv_cache *cache, const void *q, const int32_t *ring_table,
                             int32_t ring_pages, const int32_t *seq_lens, int32_t max_seq_len, int32_t batch,
                             int32_t q_len, int32_t n_heads, int32_t n_kv_heads, int32_t head_dim, float sm_scale,
                             int32_t window, void *workspace, size_t workspace_bytes, void *out, void *stream);
int memra_decode_step_window(const memra_kv_cache *cache, const void *k_new, const void *v_new, const void *q,
                             const int32_t *ring_table, int32_t ring_pages, const int32_t *seq_lens,
                             int32_t max_seq_len, int32_t batch, int32_t q_len, int32_t n_heads, int32_t n_kv_heads,
                             int32_t head_dim, float sm_scale, int32_t window, void *workspace,
                             size_t workspace_bytes, void *out, void *stream);

/* Cascade decode for a prefix that every sequence of the call shares (the
 * memra README introduction's shared-prefix serving shape: 4,860-token prompts
 * over one shared prefix at concurrency 16).  Same arguments and result as
 * memra_decode_attn / memra_decode_step, plus
 *   prefix_len   a multiple of 16, <= max_seq_len - q_len: keys 0 ..
 *                prefix_len - 1 of every sequence are the rows of the pages
 *                page_table[0][0 .. prefix_len/16 - 1]; every row of
 *                page_table must hold the same page ids there (a row that
 *                does not sets MEMRA_DEVERR_PREFIX and uses the first row's
 *                pages), and every sequence must have seq_len - q_len >=
 *                prefix_len (else MEMRA_DEVERR_BAD_SEQ_LEN).  0 runs the plain
 *                call.
 * The prefix is read and dequantized once per KV head for all query rows of
 * the call: the rows of a KV head (batch x q_len x group, 128 per tile) are
 * the M side of tensor-core MMAs.  Each sequence's own keys go through the
 * split kernel; a log-sum-exp merge joins both.  The result is the same
 * attention within the output tolerance, not byte-identical to the plain
 * call; a row's bytes depend on its own query and keys and on prefix_len
 * only, not on the rest of the batch.  head_dim 128 or 256, no window.  The
 * workspace is memra_decode_attn_cascade_workspace_bytes(...) (0 for invalid
 * sizes); memra_decode_step_cascade stores the step's rows first, as
 * memra_decode_step does. */
size_t memra_decode_attn_cascade_workspace_bytes(int32_t batch, int32_t q_len, int32_t n_heads, int32_t head_dim,
                                                 int32_t max_seq_len, int32_t prefix_len);
int memra_decode_attn_cascade(const memra_kv_cache *cache, const void *q, const int32_t *page_table,
                              int32_t max_pages_per_seq, const int32_t *seq_lens, int32_t max_seq_len,
                              int32_t prefix_len, int32_t batch, int32_t q_len, int32_t n_heads, int32_t n_kv_heads,
                              int32_t head_dim, float sm_scale, void *workspace, size_t workspace_bytes, void *out,
                              void *stream);
int memra_decode_step_cascade(const memra_kv_cache *cache, const void *k_new, const void *v_new, const void *q,
                              const int32_t *page_table, int32_t max_pages_per_seq, const int32_t *seq_lens,
                              int32_t max_seq_len, int32_t prefix_len, int32_t batch, int32_t q_len, int32_t n_heads,
                              int32_t n_kv_heads, int32_t head_dim, float sm_scale, void *workspace,
                              size_t workspace_bytes, void *out, void *stream);

/* Fixed size of the device array that memra_decode_attn_noalloc uses for the
 * split-K partials (held on every device that calls it, until exit). */
#define MEMRA_NOALLOC_SCRATCH_BYTES (16u << 20)

/* memra_decode_attn for callers that cannot allocate device memory (code
 * running inside a custom allocator or memory pool, plugins given only their
 * input and output buffers, paths that forbid allocation after start-up).
 * The memra pages have no counterpart of this call; it exists for such
 * callers.  Same arguments and results as memra_decode_attn without the
 * workspace: the partials go to a library-owned device array of
 * MEMRA_NOALLOC_SCRATCH_BYTES, so the call allocates nothing.
 *   - Returns MEMRA_ERR_WORKSPACE when memra_decode_attn_workspace_bytes(batch,
 *     q_len, n_heads, head_dim, max_seq_len) exceeds MEMRA_NOALLOC_SCRATCH_BYTES.
 *   - The first call on a device looks up the array's device address (a CUDA
 *     runtime query, no allocation) and keeps it for later calls; make that
 *     first call before any stream capture.  The kept address belongs to the
 *     device's current context: after cudaDeviceReset it is stale, so do not
 *     call this entry point again in a process that reset the device.
 *   - Every call shares the array and leaves its bytes behind; nothing in it
 *     needs to start at zero.  Calls whose kernels may overlap on the GPU
 *     (unordered streams) race on the array and must be serialized. */
int memra_decode_attn_noalloc(const memra_kv_cache *cache, const void *q, const int32_t *page_table,
                              int32_t max_pages_per_seq, const int32_t *seq_lens, int32_t max_seq_len,
                              int32_t batch, int32_t q_len, int32_t n_heads, int32_t n_kv_heads,
                              int32_t head_dim, float sm_scale, void *out, void *stream);

/* Synchronizes `stream`, reads the device status word into *flags (0 if
 * cache->status is NULL), clears it, and returns MEMRA_ERR_DEVICE if any bit
 * was set, else MEMRA_OK (or MEMRA_ERR_CUDA if the stream reported an error). */
int memra_read_status(const memra_kv_cache *cache, int32_t *flags, void *stream);

/* Static English description of a memra_status value. */
const char *memra_status_string(int status);

/* Upper bound on the split-K partials of a sequence of `seq_len` tokens
 * (ceil(seq_len / MEMRA_SPLIT_TOKENS)); the workspace is sized with it. */
int32_t memra_num_splits(int32_t seq_len);

#ifdef __cplusplus
}
#endif

#endif /* MEMRA_H */
