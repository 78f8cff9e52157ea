// Host side of the C ABI in include/memra.h: argument validation, the split
// plan, shared-memory sizing and the kernel launches.  Nothing here allocates
// device memory or synchronizes, except memra_read_status.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>

#include "cascade.cuh"
#include "decode_kernel.cuh"
#include "memra_testing.h"

using namespace memra;

namespace {

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool k_format_ok(int f) { return f == MEMRA_KV_Q8_0 || f == MEMRA_KV_FP8_E4M3 || f == MEMRA_KV_NVFP4; }
bool v_format_ok(int f) {
  return f == MEMRA_KV_Q5_1 || f == MEMRA_KV_Q4_0 || f == MEMRA_KV_FP8_E4M3 || f == MEMRA_KV_NVFP4;
}
// formats with a float32 per-tensor scale
bool scaled_format(int f) { return f == MEMRA_KV_FP8_E4M3 || f == MEMRA_KV_NVFP4; }

int check_cache(const memra_kv_cache *c) {
  if (!c) return MEMRA_ERR_INVALID_ARG;
  if (!k_format_ok(c->k_fmt) || !v_format_ok(c->v_fmt)) return MEMRA_ERR_UNSUPPORTED;
  if (c->page_size != MEMRA_PAGE_SIZE) return MEMRA_ERR_UNSUPPORTED;
  if (c->head_dim != 128 && c->head_dim != 256) return MEMRA_ERR_UNSUPPORTED;
  if (c->n_kv_heads < 1 || c->num_pages < 1) return MEMRA_ERR_INVALID_ARG;
  if (!c->k_pool || !c->v_pool || !aligned16(c->k_pool) || !aligned16(c->v_pool)) return MEMRA_ERR_INVALID_ARG;
  if (c->status && (reinterpret_cast<uintptr_t>(c->status) & 3u)) return MEMRA_ERR_INVALID_ARG;
  if (scaled_format(c->k_fmt) && !(std::isfinite(c->k_scale) && c->k_scale > 0.f)) return MEMRA_ERR_INVALID_ARG;
  if (scaled_format(c->v_fmt) && !(std::isfinite(c->v_scale) && c->v_scale > 0.f)) return MEMRA_ERR_INVALID_ARG;
  // pools larger than 2^31 segments per head are fine (size_t offsets)
  return MEMRA_OK;
}

int cuda_status(cudaError_t e) { return e == cudaSuccess ? MEMRA_OK : MEMRA_ERR_CUDA; }

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Shared memory of an SM and what the hardware reserves per resident CTA.
constexpr size_t kSmPerSm = 228 * 1024;
constexpr size_t kSmReservedPerCta = 1024;

struct Plan {
  int ngh, ngh_q, nsplit_max, num_stages, ctas_per_sm;
  size_t smem;
};

// Streaming multiprocessors of the current device (queried once per device).
int device_sms() {
  static int cached[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 1;
  if (!cached[dev]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1) n = 1;
    cached[dev] = n;
  }
  return cached[dev];
}

// Splits one long sequence gets per KV head: one wave of the GPU.
int split_target(const Plan &pl, int n_kv_heads) {
  const int t = device_sms() * pl.ctas_per_sm / (n_kv_heads > 0 ? n_kv_heads : 1);
  return t > 0 ? t : 1;
}

int warps_for(int D) { return D == 128 ? kWarpsFor<128> : kWarpsFor<256>; }

size_t merge_bytes(int D) {
  const size_t rows_w = 8, nb = D / 32;
  const size_t w = warps_for(D);
  return (w * rows_w * D + 2 * w * rows_w + w * rows_w * nb) * 4;
}

// CTAs per (split, KV head, sequence) and pipeline depth.  Every query
// position and every group of 8 query heads of a KV head gets its own CTA
// (8 rows, one per MMA column), planned from the position's own length.
// max_cta_smem caps the shared memory of one CTA (0: the kernel's CTAs per SM).
int make_plan(int D, int kf, int vf, int q_len, int group, int max_seq_len, Plan *pl, size_t max_cta_smem = 0) {
  if (q_len > MEMRA_MAX_Q_LEN || group > MEMRA_MAX_GROUP) return MEMRA_ERR_UNSUPPORTED;
  const int W = warps_for(D);
  // Pipeline depth: as many 16-token pages in flight as fit beside the other
  // CTAs of the SM, in steps of the warp count so that page i and page
  // i + depth meet the same warp.
  const size_t stage = static_cast<size_t>(k_seg_bytes(kf, D)) + v_seg_bytes(vf, D);
  const int ctas_per_sm = D == 128 ? kCtasPerSmFor<128> : kCtasPerSmFor<256>;
  const size_t qbytes = static_cast<size_t>(D == 128 ? W : 1) * (D / 32) * 512;   // Q fragments (per warp at D 128)
  size_t cta = (226 * 1024) / ctas_per_sm;
  if (max_cta_smem && max_cta_smem < cta) cta = max_cta_smem;
  const size_t fixed = 2048 + qbytes + 4 * static_cast<size_t>(kSplitPagesMax);
  const size_t budget = cta > fixed ? cta - fixed : 0;     // below the smallest plan: W stages anyway
  int ns = static_cast<int>(budget / stage) & ~(W - 1);
  if (ns > 32) ns = 32;
  if (ns < W) ns = W;
  size_t region = stage * ns;
  const size_t mb = merge_bytes(D);
  if (mb > region) region = mb;
  pl->ngh = static_cast<int>(ceil_div(group, 8));
  pl->ngh_q = pl->ngh * q_len;
  pl->nsplit_max = static_cast<int>(ceil_div(max_seq_len, kSplitTokens));
  pl->num_stages = ns;
  pl->ctas_per_sm = ctas_per_sm;
  pl->smem = region + 16 * static_cast<size_t>(ns) + 4 * static_cast<size_t>(kSplitPagesMax) + qbytes;
  return MEMRA_OK;
}

// Partials of a split pass over ranges of at most max_seq_len keys, split no
// finer than min_split tokens.
size_t workspace_parts(int32_t batch, int32_t q_len, int32_t n_heads, int32_t head_dim, int32_t max_seq_len,
                       size_t *lse_offset, int min_split = kSplitTokens) {
  const size_t rows = static_cast<size_t>(batch) * q_len * n_heads;
  const size_t ns = static_cast<size_t>(ceil_div(max_seq_len, min_split));
  size_t o_bytes = rows * ns * head_dim * sizeof(float);
  o_bytes = (o_bytes + 255) & ~static_cast<size_t>(255);
  if (lse_offset) *lse_offset = o_bytes;
  return o_bytes + rows * ns * sizeof(float);
}

struct DecodeArgs {
  const memra_kv_cache *cache;
  const void *q;
  const int32_t *page_table;
  int32_t max_pages_per_seq;
  const int32_t *seq_lens;
  int32_t max_seq_len, batch, q_len, n_heads, n_kv_heads, head_dim;
  float sm_scale;
  void *workspace;
  size_t workspace_bytes;
  void *out;
  int32_t window;     // sliding window (tokens); > 0 also makes page_table rows rings
  int32_t prefix = 0; // cascade: tokens shared by every sequence, attended by the prefix pass
  // test hooks of the bounded waits (memra_testing.h): 0 = the normal limit / no short page
  uint64_t test_wait_ns = 0;
  int32_t test_extra_tx = 0;
};

// Workspace of a cascade call: the split kernel's partials over each
// sequence's own keys (at most max_seq_len - prefix of them), then the prefix
// pass's partials, [rows][chunks][D] floats and [rows][chunks] lse.
size_t cascade_parts(int32_t batch, int32_t q_len, int32_t n_heads, int32_t head_dim, int32_t max_seq_len,
                     int32_t prefix, size_t *suf_lse, size_t *pre_o, size_t *pre_lse) {
  size_t sl = 0;
  size_t suf = workspace_parts(batch, q_len, n_heads, head_dim, max_seq_len - prefix, &sl, kCascadeSplitTokens);
  suf = (suf + 255) & ~static_cast<size_t>(255);
  const size_t rows = static_cast<size_t>(batch) * q_len * n_heads;
  const size_t nch = prefix > 0 ? static_cast<size_t>(ceil_div(prefix, cascade_chunk_tokens(head_dim))) : 0;
  size_t o = rows * nch * head_dim * sizeof(float);
  o = (o + 255) & ~static_cast<size_t>(255);
  if (suf_lse) *suf_lse = sl;
  if (pre_o) *pre_o = suf;
  if (pre_lse) *pre_lse = suf + o;
  return suf + o + rows * nch * sizeof(float);
}

// Longest key range any position of the call can have: the window (+ the part
// of its first page before it) or the whole context.
int64_t longest_range(int32_t max_seq_len, int32_t window) {
  return window > 0 ? std::min<int64_t>(max_seq_len, static_cast<int64_t>(window) + kPage - 1) : max_seq_len;
}

int check_decode(const DecodeArgs &a) {
  int st = check_cache(a.cache);
  if (st) return st;
  if (a.batch < 0 || a.q_len < 1 || a.n_heads < 1 || a.max_seq_len < 0 || a.max_pages_per_seq < 0)
    return MEMRA_ERR_INVALID_ARG;
  if (a.n_kv_heads != a.cache->n_kv_heads || a.head_dim != a.cache->head_dim) return MEMRA_ERR_INVALID_ARG;
  if (a.n_heads % a.n_kv_heads) return MEMRA_ERR_INVALID_ARG;
  if (a.q_len > MEMRA_MAX_Q_LEN || a.n_heads / a.n_kv_heads > MEMRA_MAX_GROUP || a.batch > 65535 ||
      a.n_kv_heads > 65535)
    return MEMRA_ERR_UNSUPPORTED;
  if (!std::isfinite(a.sm_scale)) return MEMRA_ERR_INVALID_ARG;
  if (a.batch == 0) return MEMRA_OK;
  if (!a.q || !a.page_table || !a.seq_lens || !a.out) return MEMRA_ERR_INVALID_ARG;
  if (!aligned16(a.q) || !aligned16(a.out) || (reinterpret_cast<uintptr_t>(a.page_table) & 3u) ||
      (reinterpret_cast<uintptr_t>(a.seq_lens) & 3u))
    return MEMRA_ERR_INVALID_ARG;
  if (a.max_pages_per_seq < 1) return MEMRA_ERR_INVALID_ARG;
  if (a.window < 0) return MEMRA_ERR_INVALID_ARG;
  // a ring must hold every page that the window of any query row reaches
  if (a.window > 0 && a.max_pages_per_seq < (static_cast<int64_t>(a.window) + a.q_len - 2) / kPage + 2)
    return MEMRA_ERR_INVALID_ARG;
  if (a.prefix < 0 || a.prefix % kPage) return MEMRA_ERR_INVALID_ARG;
  if (a.prefix > 0) {
    // every query row must see the whole prefix; its pages must be in the table
    if (a.window > 0) return MEMRA_ERR_UNSUPPORTED;
    if (a.prefix > static_cast<int64_t>(a.max_seq_len) - a.q_len || a.prefix / kPage > a.max_pages_per_seq)
      return MEMRA_ERR_INVALID_ARG;
    const int64_t rows = static_cast<int64_t>(a.batch) * a.q_len * (a.n_heads / a.n_kv_heads);
    if (ceil_div(rows, 128) > 65535) return MEMRA_ERR_UNSUPPORTED;
  }
  const size_t need = a.prefix > 0 ? cascade_parts(a.batch, a.q_len, a.n_heads, a.head_dim, a.max_seq_len, a.prefix,
                                                   nullptr, nullptr, nullptr)
                                   : workspace_parts(a.batch, a.q_len, a.n_heads, a.head_dim, a.max_seq_len, nullptr);
  if (a.workspace_bytes < need) return MEMRA_ERR_WORKSPACE;
  if (need > 0 && (!a.workspace || !aligned16(a.workspace))) return MEMRA_ERR_INVALID_ARG;
  return MEMRA_OK;
}

// Chunks per prefix-pass CTA of a cascade call: few enough CTAs per KV head
// that one row tile's fit one wave of the pass, at least
// kCascadeMinChunksPerCta and never more than kCascadeMaxChunksPerCta chunks
// each.  Depends on the prefix, head_dim, formats, KV heads and the device
// only.
int cascade_cpc(int32_t prefix, int32_t head_dim, int kf, int vf, int32_t n_kv_heads, int *cpc) {
  int wave = 1;
  if (cascade_wave(head_dim, kf, vf, &wave) != cudaSuccess) return MEMRA_ERR_CUDA;
  const int64_t n_chunks = ceil_div(prefix, cascade_chunk_tokens(head_dim));
  const int64_t target = std::max<int64_t>(1, wave / n_kv_heads);
  const int64_t floor = std::min<int64_t>(kCascadeMinChunksPerCta, std::max<int64_t>(n_chunks, 1));
  *cpc = static_cast<int>(std::min<int64_t>(std::max<int64_t>(ceil_div(n_chunks, target), floor),
                                            kCascadeMaxChunksPerCta));
  return MEMRA_OK;
}

// k_new / v_new: the fused append's rows, or null for attention alone.
int run_partials(const DecodeArgs &a, const void *k_new, const void *v_new, cudaStream_t st) {
  const memra_kv_cache &c = *a.cache;
  Plan pl;
  const int group = a.n_heads / a.n_kv_heads;
  // A cascade call's own-key pass runs beside the prefix pass: where a CTA
  // with the pass's shallowest pipeline fits an SM beside a prefix CTA, its
  // shared memory is capped to that room, so that both share the SM.  Where
  // none fits (the warp-specialized head_dim 128 prefix CTA fills its SM),
  // the own-key CTAs run on the other SMs and keep the full pipeline: capped,
  // they would hold one page per warp and wait a memory round trip per page.
  size_t cap = 0;
  if (a.prefix > 0) {
    int cpc = 1;
    int rc0 = cascade_cpc(a.prefix, a.head_dim, c.k_fmt, c.v_fmt, a.n_kv_heads, &cpc);
    if (rc0) return rc0;
    const int pre_per_sm = cascade_ctas_per_sm(a.head_dim);
    const size_t pre = pre_per_sm * static_cast<size_t>(cascade_smem_bytes(
                                        a.head_dim, k_seg_bytes(c.k_fmt, a.head_dim), v_seg_bytes(c.v_fmt, a.head_dim), cpc));
    const size_t used = kSmReservedPerCta * (1 + pre_per_sm) + pre;
    cap = used < kSmPerSm ? kSmPerSm - used : 1;
    Plan smallest;
    int rc1 = make_plan(a.head_dim, c.k_fmt, c.v_fmt, a.q_len, group, a.max_seq_len, &smallest, 1);
    if (rc1) return rc1;
    if (smallest.smem > cap) cap = 0;
  }
  int rc = make_plan(a.head_dim, c.k_fmt, c.v_fmt, a.q_len, group, a.max_seq_len, &pl, cap);
  if (rc) return rc;
  // keys this pass covers: all of them, or (cascade) those from the prefix end on
  const int32_t range_max = a.max_seq_len - a.prefix;
  const int min_split = a.prefix > 0 ? kCascadeSplitTokens : kSplitTokens;
  const int nsplit_max = static_cast<int>(ceil_div(range_max, min_split));
  if (nsplit_max == 0) return MEMRA_OK;       // every sequence is empty; the combine writes zeros
  size_t lse_off = 0;
  workspace_parts(a.batch, a.q_len, a.n_heads, a.head_dim, range_max, &lse_off, min_split);
  DecodeParams p;
  p.k_pool = static_cast<const uint8_t *>(c.k_pool);
  p.v_pool = static_cast<const uint8_t *>(c.v_pool);
  p.q = static_cast<const __half *>(a.q);
  p.page_table = a.page_table;
  p.seq_lens = a.seq_lens;
  p.out = static_cast<__half *>(a.out);
  p.o_part = static_cast<float *>(a.workspace);
  p.lse_part = reinterpret_cast<float *>(static_cast<uint8_t *>(a.workspace) + lse_off);
  p.status = c.status;
  p.k_new = static_cast<const __half *>(k_new);
  p.v_new = static_cast<const __half *>(v_new);
  p.n_kv_heads = c.n_kv_heads;
  p.num_pages = c.num_pages;
  p.max_pages = a.max_pages_per_seq;
  p.max_seq_len = a.max_seq_len;
  p.q_len = a.q_len;
  p.n_heads = a.n_heads;
  p.group = group;
  p.window = a.window;
  p.skip = a.prefix;
  p.ring = a.window > 0 ? 1 : 0;
  p.ngh = pl.ngh;
  p.ngh_q = pl.ngh_q;
  p.nsplit_max = nsplit_max;
  p.num_stages = pl.num_stages;
  p.split_target = split_target(pl, c.n_kv_heads);
  const float k_scale = scaled_format(c.k_fmt) ? c.k_scale : 1.f;
  p.scale_log2 = a.sm_scale * k_scale * 1.4426950408889634f;
  p.v_scale = scaled_format(c.v_fmt) ? c.v_scale : 1.f;
  p.k_scale = c.k_scale;
  p.page_wait_ns = a.test_wait_ns ? a.test_wait_ns : kWaitLimitNs;
  p.test_extra_tx = a.test_extra_tx;
  // no position has more splits than min(ceil(L/min), max(target, ceil(L/8192))), L its key range
  const int64_t L = a.prefix > 0 ? range_max : longest_range(a.max_seq_len, a.window);
  const int64_t most = std::min<int64_t>(ceil_div(L, min_split),
                                         std::max<int64_t>(p.split_target, ceil_div(L, kSplitTokensMax)));
  // x: split-major, then query position and head group (the CTAs that read
  // the same pages run side by side and share them through L2)
  const dim3 grid(static_cast<unsigned>(most * pl.ngh_q), static_cast<unsigned>(c.n_kv_heads),
                  static_cast<unsigned>(a.batch));
  const cudaError_t e = a.head_dim == 128 ? launch_decode_d128(c.k_fmt, c.v_fmt, p, grid, pl.smem, st)
                                          : launch_decode_d256(c.k_fmt, c.v_fmt, p, grid, pl.smem, st);
  return cuda_status(e);
}

int run_combine(const memra_kv_cache *c, const int32_t *seq_lens, int32_t max_seq_len, int32_t max_pages,
                int32_t batch, int32_t q_len, int32_t n_heads, int32_t head_dim, int32_t window,
                const void *workspace, void *out, cudaStream_t st) {
  size_t lse_off = 0;
  workspace_parts(batch, q_len, n_heads, head_dim, max_seq_len, &lse_off);
  CombineParams p;
  p.seq_lens = seq_lens;
  p.o_part = static_cast<const float *>(workspace);
  p.lse_part = reinterpret_cast<const float *>(static_cast<const uint8_t *>(workspace) + lse_off);
  p.out = static_cast<__half *>(out);
  p.status = c->status;
  p.rows = batch * q_len * n_heads;
  p.q_len = q_len;
  p.n_heads = n_heads;
  p.max_seq_len = max_seq_len;
  p.max_pages = max_pages;
  p.nsplit_max = static_cast<int>(ceil_div(max_seq_len, kSplitTokens));
  p.window = window;
  p.ring = window > 0 ? 1 : 0;
  Plan pl;
  int rc = make_plan(head_dim, c->k_fmt, c->v_fmt, q_len, n_heads / c->n_kv_heads, max_seq_len, &pl);
  if (rc) return rc;
  p.split_target = split_target(pl, c->n_kv_heads);
  return cuda_status(launch_combine(head_dim, p, st));
}

}  // namespace

extern "C" {

size_t memra_kv_segment_bytes(int32_t fmt, int32_t is_v, int32_t head_dim) {
  if (head_dim != 128 && head_dim != 256) return 0;
  if (is_v == 0) return k_format_ok(fmt) ? static_cast<size_t>(k_seg_bytes(fmt, head_dim)) : 0;
  if (is_v == 1) return v_format_ok(fmt) ? static_cast<size_t>(v_seg_bytes(fmt, head_dim)) : 0;
  return 0;
}

size_t memra_kv_pool_bytes(int32_t fmt, int32_t is_v, int32_t num_pages, int32_t page_size, int32_t n_kv_heads,
                           int32_t head_dim) {
  if (page_size != MEMRA_PAGE_SIZE || num_pages < 1 || n_kv_heads < 1) return 0;
  return memra_kv_segment_bytes(fmt, is_v, head_dim) * static_cast<size_t>(num_pages) * n_kv_heads;
}

int memra_kv_append(const memra_kv_cache *cache, const void *k, const void *v, const int32_t *slot_mapping,
                    int32_t n_tok, void *stream) {
  int st = check_cache(cache);
  if (st) return st;
  if (n_tok < 0) return MEMRA_ERR_INVALID_ARG;
  if (n_tok == 0) return MEMRA_OK;
  if (!k || !v || !slot_mapping || !aligned16(k) || !aligned16(v) ||
      (reinterpret_cast<uintptr_t>(slot_mapping) & 3u))
    return MEMRA_ERR_INVALID_ARG;
  return cuda_status(launch_kv_append(*cache, k, v, slot_mapping, n_tok, static_cast<cudaStream_t>(stream)));
}

size_t memra_decode_attn_workspace_bytes(int32_t batch, int32_t q_len, int32_t n_heads, int32_t head_dim,
                                         int32_t max_seq_len) {
  if (batch < 0 || q_len < 1 || n_heads < 1 || (head_dim != 128 && head_dim != 256) || max_seq_len < 0) return 0;
  return workspace_parts(batch, q_len, n_heads, head_dim, max_seq_len, nullptr);
}

int memra_decode_attn_partials(const memra_kv_cache *cache, const void *q, const int32_t *page_table,
                               int32_t max_pages_per_seq, const int32_t *seq_lens, int32_t max_seq_len, int32_t batch,
                               int32_t q_len, int32_t n_heads, int32_t n_kv_heads, int32_t head_dim, float sm_scale,
                               void *workspace, size_t workspace_bytes, void *out, void *stream) {
  DecodeArgs a{cache, q, page_table, max_pages_per_seq, seq_lens, max_seq_len, batch, q_len, n_heads,
               n_kv_heads, head_dim, sm_scale, workspace, workspace_bytes, out, 0};
  int st = check_decode(a);
  if (st || batch == 0) return st;
  return run_partials(a, nullptr, nullptr, static_cast<cudaStream_t>(stream));
}

int memra_decode_attn_combine(const memra_kv_cache *cache, const int32_t *seq_lens, int32_t max_seq_len,
                              int32_t max_pages_per_seq, int32_t batch, int32_t q_len, int32_t n_heads,
                              int32_t head_dim, const void *workspace, size_t workspace_bytes, void *out,
                              void *stream) {
  int st = check_cache(cache);
  if (st) return st;
  if (batch < 0 || q_len < 1 || n_heads < 1 || max_seq_len < 0 || head_dim != cache->head_dim ||
      max_pages_per_seq < 0 || n_heads % cache->n_kv_heads)
    return MEMRA_ERR_INVALID_ARG;
  if (batch == 0) return MEMRA_OK;
  if (!seq_lens || !out || !aligned16(out)) return MEMRA_ERR_INVALID_ARG;
  const size_t need = workspace_parts(batch, q_len, n_heads, head_dim, max_seq_len, nullptr);
  if (workspace_bytes < need) return MEMRA_ERR_WORKSPACE;
  if (need > 0 && (!workspace || !aligned16(workspace))) return MEMRA_ERR_INVALID_ARG;
  return run_combine(cache, seq_lens, max_seq_len, max_pages_per_seq, batch, q_len, n_heads, head_dim, 0, workspace,
                     out, static_cast<cudaStream_t>(stream));
}

}  // extern "C"

namespace {

// Split pass (with the fused append when k_new / v_new are given), then the combine.
int decode_both_passes(const DecodeArgs &a, const void *k_new, const void *v_new, void *stream) {
  int st = check_decode(a);
  if (st || a.batch == 0) return st;
  if (k_new || v_new) {
    if (!k_new || !v_new || !aligned16(k_new) || !aligned16(v_new)) return MEMRA_ERR_INVALID_ARG;
    if (a.max_seq_len < a.q_len) return MEMRA_ERR_INVALID_ARG;     // no sequence can hold the new rows
  }
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  st = run_partials(a, k_new, v_new, s);
  if (st) return st;
  // Every row fits one split (no split is shorter than kSplitTokens): the
  // split pass wrote every row, zeros included, and there is nothing to merge.
  if (a.max_seq_len > 0 && a.max_seq_len <= kSplitTokens) return MEMRA_OK;
  return run_combine(a.cache, a.seq_lens, a.max_seq_len, a.max_pages_per_seq, a.batch, a.q_len, a.n_heads,
                     a.head_dim, a.window, a.workspace, a.out, s);
}

// Cascade: the prefix pass (tcgen05), the split kernel over each sequence's
// own keys (with the fused append when k_new / v_new are given), the merge.
int cascade_passes(const DecodeArgs &a, const void *k_new, const void *v_new, void *stream) {
  if (a.prefix == 0) return decode_both_passes(a, k_new, v_new, stream);
  int st = check_decode(a);
  if (st || a.batch == 0) return st;
  if (k_new || v_new) {
    if (!k_new || !v_new || !aligned16(k_new) || !aligned16(v_new)) return MEMRA_ERR_INVALID_ARG;
  }
  const memra_kv_cache &c = *a.cache;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  size_t suf_lse = 0, pre_o = 0, pre_lse = 0;
  cascade_parts(a.batch, a.q_len, a.n_heads, a.head_dim, a.max_seq_len, a.prefix, &suf_lse, &pre_o, &pre_lse);
  uint8_t *ws = static_cast<uint8_t *>(a.workspace);
  const int group = a.n_heads / a.n_kv_heads;
  const int n_chunks = static_cast<int>(ceil_div(a.prefix, cascade_chunk_tokens(a.head_dim)));

  CascadeParams cp;
  cp.k_pool = static_cast<const uint8_t *>(c.k_pool);
  cp.v_pool = static_cast<const uint8_t *>(c.v_pool);
  cp.q = static_cast<const __half *>(a.q);
  cp.page_table = a.page_table;
  cp.seq_lens = a.seq_lens;
  cp.status = c.status;
  cp.o_pre = reinterpret_cast<float *>(ws + pre_o);
  cp.lse_pre = reinterpret_cast<float *>(ws + pre_lse);
  cp.batch = a.batch;
  cp.q_len = a.q_len;
  cp.n_heads = a.n_heads;
  cp.group = group;
  cp.n_kv_heads = a.n_kv_heads;
  cp.num_pages = c.num_pages;
  cp.max_pages = a.max_pages_per_seq;
  cp.prefix_len = a.prefix;
  cp.n_chunks = n_chunks;
  st = cascade_cpc(a.prefix, a.head_dim, c.k_fmt, c.v_fmt, a.n_kv_heads, &cp.cpc);
  if (st) return st;
  // staged values: q8_0 / q5_1 / q4_0 at half size, fp8 / NVFP4 without their tensor scale
  const float k_post = c.k_fmt == MEMRA_KV_Q8_0 ? 2.f : c.k_scale;
  cp.scale_log2 = a.sm_scale * k_post * 1.4426950408889634f;
  cp.v_post = scaled_format(c.v_fmt) ? c.v_scale : 2.f;
  st = cuda_status(launch_cascade_prefix(a.head_dim, c.k_fmt, c.v_fmt, cp, s));
  if (st) return st;

  st = run_partials(a, k_new, v_new, s);
  if (st) return st;

  Plan pl;
  st = make_plan(a.head_dim, c.k_fmt, c.v_fmt, a.q_len, group, a.max_seq_len, &pl);
  if (st) return st;
  CascadeCombineParams mp;
  mp.seq_lens = a.seq_lens;
  mp.o_pre = cp.o_pre;
  mp.lse_pre = cp.lse_pre;
  mp.o_suf = reinterpret_cast<const float *>(ws);
  mp.lse_suf = reinterpret_cast<const float *>(ws + suf_lse);
  mp.out = static_cast<__half *>(a.out);
  mp.status = c.status;
  mp.rows = a.batch * a.q_len * a.n_heads;
  mp.q_len = a.q_len;
  mp.n_heads = a.n_heads;
  mp.max_seq_len = a.max_seq_len;
  mp.max_pages = a.max_pages_per_seq;
  mp.nsplit_max = static_cast<int>(ceil_div(a.max_seq_len - a.prefix, kCascadeSplitTokens));
  mp.split_target = split_target(pl, c.n_kv_heads);
  mp.prefix_len = a.prefix;
  mp.n_parts = cp.n_parts;
  return cuda_status(launch_cascade_combine(a.head_dim, mp, s));
}

}  // namespace

extern "C" {

size_t memra_decode_attn_cascade_workspace_bytes(int32_t batch, int32_t q_len, int32_t n_heads, int32_t head_dim,
                                                 int32_t max_seq_len, int32_t prefix_len) {
  if (batch < 0 || q_len < 1 || n_heads < 1 || (head_dim != 128 && head_dim != 256) || max_seq_len < 0 ||
      prefix_len < 0 || prefix_len % kPage || prefix_len > max_seq_len)
    return 0;
  return cascade_parts(batch, q_len, n_heads, head_dim, max_seq_len, prefix_len, nullptr, nullptr, nullptr);
}

int memra_decode_attn_cascade(const memra_kv_cache *cache, const void *q, const int32_t *page_table,
                              int32_t max_pages_per_seq, const int32_t *seq_lens, int32_t max_seq_len,
                              int32_t prefix_len, int32_t batch, int32_t q_len, int32_t n_heads, int32_t n_kv_heads,
                              int32_t head_dim, float sm_scale, void *workspace, size_t workspace_bytes, void *out,
                              void *stream) {
  const DecodeArgs a{cache, q, page_table, max_pages_per_seq, seq_lens, max_seq_len, batch, q_len, n_heads,
                     n_kv_heads, head_dim, sm_scale, workspace, workspace_bytes, out, 0, prefix_len};
  return cascade_passes(a, nullptr, nullptr, stream);
}

int memra_decode_step_cascade(const memra_kv_cache *cache, const void *k_new, const void *v_new, const void *q,
                              const int32_t *page_table, int32_t max_pages_per_seq, const int32_t *seq_lens,
                              int32_t max_seq_len, int32_t prefix_len, int32_t batch, int32_t q_len, int32_t n_heads,
                              int32_t n_kv_heads, int32_t head_dim, float sm_scale, void *workspace,
                              size_t workspace_bytes, void *out, void *stream) {
  if (!k_new || !v_new) return MEMRA_ERR_INVALID_ARG;
  const DecodeArgs a{cache, q, page_table, max_pages_per_seq, seq_lens, max_seq_len, batch, q_len, n_heads,
                     n_kv_heads, head_dim, sm_scale, workspace, workspace_bytes, out, 0, prefix_len};
  return cascade_passes(a, k_new, v_new, stream);
}

int memra_decode_attn(const memra_kv_cache *cache, const void *q, const int32_t *page_table,
                      int32_t max_pages_per_seq, const int32_t *seq_lens, int32_t max_seq_len, int32_t batch,
                      int32_t q_len, int32_t n_heads, int32_t n_kv_heads, int32_t head_dim, float sm_scale,
                      void *workspace, size_t workspace_bytes, void *out, void *stream) {
  const DecodeArgs a{cache, q, page_table, max_pages_per_seq, seq_lens, max_seq_len, batch, q_len, n_heads,
                     n_kv_heads, head_dim, sm_scale, workspace, workspace_bytes, out, 0};
  return decode_both_passes(a, nullptr, nullptr, stream);
}

int memra_decode_step(const memra_kv_cache *cache, const void *k_new, const void *v_new, const void *q,
                      const int32_t *page_table, int32_t max_pages_per_seq, const int32_t *seq_lens,
                      int32_t max_seq_len, int32_t batch, int32_t q_len, int32_t n_heads, int32_t n_kv_heads,
                      int32_t head_dim, float sm_scale, void *workspace, size_t workspace_bytes, void *out,
                      void *stream) {
  if (!k_new || !v_new) return MEMRA_ERR_INVALID_ARG;
  const DecodeArgs a{cache, q, page_table, max_pages_per_seq, seq_lens, max_seq_len, batch, q_len, n_heads,
                     n_kv_heads, head_dim, sm_scale, workspace, workspace_bytes, out, 0};
  return decode_both_passes(a, k_new, v_new, stream);
}

int memra_decode_attn_window(const memra_kv_cache *cache, const void *q, const int32_t *ring_table,
                             int32_t ring_pages, const int32_t *seq_lens, int32_t max_seq_len, int32_t batch,
                             int32_t q_len, int32_t n_heads, int32_t n_kv_heads, int32_t head_dim, float sm_scale,
                             int32_t window, void *workspace, size_t workspace_bytes, void *out, void *stream) {
  if (window < 1) return MEMRA_ERR_INVALID_ARG;
  const DecodeArgs a{cache, q, ring_table, ring_pages, seq_lens, max_seq_len, batch, q_len, n_heads,
                     n_kv_heads, head_dim, sm_scale, workspace, workspace_bytes, out, window};
  return decode_both_passes(a, nullptr, nullptr, stream);
}

int memra_decode_step_window(const memra_kv_cache *cache, const void *k_new, const void *v_new, const void *q,
                             const int32_t *ring_table, int32_t ring_pages, const int32_t *seq_lens,
                             int32_t max_seq_len, int32_t batch, int32_t q_len, int32_t n_heads, int32_t n_kv_heads,
                             int32_t head_dim, float sm_scale, int32_t window, void *workspace,
                             size_t workspace_bytes, void *out, void *stream) {
  if (window < 1 || !k_new || !v_new) return MEMRA_ERR_INVALID_ARG;
  const DecodeArgs a{cache, q, ring_table, ring_pages, seq_lens, max_seq_len, batch, q_len, n_heads,
                     n_kv_heads, head_dim, sm_scale, workspace, workspace_bytes, out, window};
  return decode_both_passes(a, k_new, v_new, stream);
}

int memra_read_status(const memra_kv_cache *cache, int32_t *flags, void *stream) {
  if (!cache || !flags) return MEMRA_ERR_INVALID_ARG;
  *flags = 0;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return MEMRA_ERR_CUDA;
  if (!cache->status) return MEMRA_OK;
  int32_t host = 0;
  if (cudaMemcpyAsync(&host, cache->status, sizeof(int32_t), cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return MEMRA_ERR_CUDA;
  if (cudaMemsetAsync(cache->status, 0, sizeof(int32_t), s) != cudaSuccess) return MEMRA_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return MEMRA_ERR_CUDA;
  *flags = host;
  return host ? MEMRA_ERR_DEVICE : MEMRA_OK;
}

const char *memra_status_string(int status) {
  switch (status) {
    case MEMRA_OK: return "ok";
    case MEMRA_ERR_INVALID_ARG: return "invalid argument";
    case MEMRA_ERR_UNSUPPORTED: return "unsupported configuration";
    case MEMRA_ERR_WORKSPACE: return "workspace too small";
    case MEMRA_ERR_CUDA: return "CUDA error";
    case MEMRA_ERR_DEVICE: return "the device flagged an error (see the status bits)";
    default: return "unknown status";
  }
}

int32_t memra_num_splits(int32_t seq_len) {
  return seq_len <= 0 ? 0 : static_cast<int32_t>(ceil_div(seq_len, kSplitTokens));
}

}  // extern "C"

// ------------------------------------------------------------ test hooks --
// memra_testing.h: the decode call with a shortened page-wait limit and one
// page whose wait cannot complete, to drive the bounded-wait path on a GPU.
extern "C" int memra_testing_decode_attn_short_page(const memra_kv_cache *cache, const void *q,
                                                    const int32_t *page_table, int32_t max_pages_per_seq,
                                                    const int32_t *seq_lens, int32_t max_seq_len, int32_t batch,
                                                    int32_t q_len, int32_t n_heads, int32_t n_kv_heads,
                                                    int32_t head_dim, float sm_scale, void *workspace,
                                                    size_t workspace_bytes, void *out, uint64_t page_wait_ns,
                                                    void *stream) {
  if (page_wait_ns == 0 || page_wait_ns > kWaitLimitNs) return MEMRA_ERR_INVALID_ARG;
  DecodeArgs a{cache, q, page_table, max_pages_per_seq, seq_lens, max_seq_len, batch, q_len, n_heads,
               n_kv_heads, head_dim, sm_scale, workspace, workspace_bytes, out, 0};
  a.test_wait_ns = page_wait_ns;
  a.test_extra_tx = 16;
  return decode_both_passes(a, nullptr, nullptr, stream);
}

// memra_testing.h: the quantizer's division by a scale (kv_quant.cuh) against
// the IEEE quotient, for every finite fp16 dividend and the given scales.
namespace {
__global__ void scale_division_check_kernel(const float *scales, unsigned long long *mismatches) {
  const float s = scales[blockIdx.y];
  const float r = __frcp_rn(s);
  unsigned long long bad = 0;
  for (int bits = blockIdx.x * blockDim.x + threadIdx.x; bits < 65536; bits += gridDim.x * blockDim.x) {
    const float x = __half2float(__ushort_as_half(static_cast<unsigned short>(bits)));
    if (!isfinite(x)) continue;
    if (__float_as_uint(memra::div_by_scale(x, s, r)) != __float_as_uint(__fdiv_rn(x, s))) ++bad;
  }
  if (bad) atomicAdd(mismatches, bad);
}
}  // namespace

extern "C" int memra_testing_scale_division_mismatches(const float *scales, int32_t n_scales,
                                                       unsigned long long *mismatches, void *stream) {
  if (!scales || !mismatches || n_scales < 1 || n_scales > 65535) return MEMRA_ERR_INVALID_ARG;
  scale_division_check_kernel<<<dim3(16, static_cast<unsigned>(n_scales)), 256, 0, static_cast<cudaStream_t>(stream)>>>(
      scales, mismatches);
  return cudaGetLastError() == cudaSuccess ? MEMRA_OK : MEMRA_ERR_CUDA;
}
