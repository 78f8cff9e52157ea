// Cascade decode over a prefix shared by every sequence of a call: the
// parameters of its two kernels (the prefix pass and the merge) and their
// launchers.  The sequences' own keys go through the split kernel with
// DecodeParams::skip = the prefix length.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "memra_device.cuh"

namespace memra {

// Prefix tokens of one chunk (the N of the score MMA), and prefix-pass CTAs
// per SM: one either way (the warp-specialized head_dim 128 pass fills the
// SM's shared memory; the head_dim 256 pass needs more than half of it).
__host__ __device__ constexpr int cascade_chunk_tokens(int D) { return D == 128 ? 64 : 64; }
__host__ __device__ constexpr int cascade_ctas_per_sm(int D) { return D == 128 ? 1 : 1; }

struct CascadeParams {
  const uint8_t *k_pool;
  const uint8_t *v_pool;
  const __half *q;
  const int32_t *page_table;
  const int32_t *seq_lens;
  int32_t *status;
  float *o_pre;       // [batch * q_len * n_heads][n_parts][D], row id (b * q_len + i) * n_heads + h
  float *lse_pre;     // [batch * q_len * n_heads][n_parts]
  int batch, q_len, n_heads, group, n_kv_heads, num_pages, max_pages, prefix_len, n_chunks;
  int cpc;            // chunks per CTA (1 .. kCascadeMaxChunksPerCta)
  int n_parts;        // prefix partials per row: the CTAs per (KV head, row tile), set by the launcher
  float scale_log2;   // sm_scale * (post-scale of the staged K values) * log2(e)
  float v_post;       // post-scale of the staged V values
};

struct CascadeCombineParams {
  const int32_t *seq_lens;
  const float *o_pre;
  const float *lse_pre;
  const float *o_suf;     // the split kernel's partials of the keys from the prefix end on
  const float *lse_suf;
  __half *out;
  int32_t *status;
  int rows, q_len, n_heads, max_seq_len, max_pages, nsplit_max, split_target, prefix_len;
  int n_parts;            // prefix partials per row (CascadeParams::n_parts of the prefix pass)
};

// Chunks one prefix-pass CTA loops over at most, and at least (unless the
// prefix is shorter).  The floor keeps a CTA's fixed costs (page ids, the Q
// tile, the first copies, the output rows) to a fraction of its time, and on
// a short prefix it leaves SMs free for the call's own-key pass, which then
// runs beside the prefix pass instead of after it.
constexpr int kCascadeMaxChunksPerCta = 64;
constexpr int kCascadeMinChunksPerCta = 3;

// Shared memory of one prefix-pass CTA for head_dim D, the formats' segment
// bytes and cpc chunks per CTA: the Q tile, one half-chunk of K^ and of V^T
// (hi and lo parts), the raw pages (two buffers when the CTA loops), the
// softmax exchange, the page ids, the barriers.
// At head_dim 256 the request is at least 155 KiB, so that no other prefix-pass
// CTA (and its tensor memory) fits beside it.  At head_dim 128 (the
// warp-specialized pass): the Q tile, two K^ and two V^T chunk buffers (hi and
// lo parts), two P buffers, two raw page buffers, the page ids, the barriers.
__host__ __device__ constexpr uint32_t cascade_smem_plan(int D, int kseg, int vseg, int cpc) {
  return D == 128
             ? 128u * D * 2 + 8u * cascade_chunk_tokens(D) * D * 2 + 2u * 128u * cascade_chunk_tokens(D) * 2 +
                   2u * static_cast<uint32_t>(cascade_chunk_tokens(D) / MEMRA_PAGE_SIZE) * (kseg + vseg) +
                   4u * static_cast<uint32_t>(cascade_chunk_tokens(D) / MEMRA_PAGE_SIZE) * cpc + 192u
             : 128u * D * 2 + 2u * cascade_chunk_tokens(D) * D * 2 +
                   (cpc > 1 ? 2u : 1u) * static_cast<uint32_t>(cascade_chunk_tokens(D) / MEMRA_PAGE_SIZE) *
                       (kseg + vseg) +
                   4u * 128u * 4u + 4u * static_cast<uint32_t>(cascade_chunk_tokens(D) / MEMRA_PAGE_SIZE) * cpc + 64u;
}
__host__ __device__ constexpr uint32_t cascade_smem_bytes(int D, int kseg, int vseg, int cpc) {
  return D == 256 && cascade_smem_plan(D, kseg, vseg, cpc) < 155u * 1024u ? 155u * 1024u
                                                                           : cascade_smem_plan(D, kseg, vseg, cpc);
}

// Tensor-memory columns of one prefix-pass CTA, a power of two: at head_dim
// 128, O and two score buffers (256); at 256, O and one score buffer (512).
// The hardware places CTAs by registers and shared memory, not by tensor
// memory, so any mix of prefix-pass CTAs that fits an SM by shared memory
// must fit its 512 columns: here, one CTA of either kind (>= 205 KB and >=
// 155 KB).  A CTA that found the columns taken would wait in its allocation.
__host__ __device__ constexpr uint32_t cascade_tmem_cols(int D) { return D == 128 ? 256u : 512u; }

// The CTAs one wave of the prefix pass holds on this device (independent of
// the batch).
cudaError_t cascade_wave(int D, int kf, int vf, int *wave_ctas);

// Fills p.n_parts (one partial per CTA of a row tile) and launches.
cudaError_t launch_cascade_prefix(int D, int kf, int vf, CascadeParams &p, cudaStream_t st);
cudaError_t launch_cascade_combine(int D, const CascadeCombineParams &p, cudaStream_t st);

}  // namespace memra
