// K3: log-sum-exp combine of the split-K partials.
//
// For a query row whose sequence spans several 1024-token splits, the split
// kernel left (o_s = O_s / l_s, lse_s = m_s + log2 l_s) per split.  The exact
// merge is  out = sum_s 2^(lse_s - M) o_s / sum_s 2^(lse_s - M),  M = max lse_s
// (splits with no visible key have lse = -inf and weight 0).  One warp per
// row; each lane owns D/32 consecutive outputs, so every split's partial is
// one coalesced 512 B (D 128) or 1 KiB (D 256) read.
#include <cuda_runtime.h>

#include "decode_kernel.cuh"

namespace memra {

template <int D>
__global__ void __launch_bounds__(128) combine_kernel(const CombineParams p) {
  constexpr int PER = D / 32;
  const int row = blockIdx.x * 4 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= p.rows) return;
  const int b = row / (p.q_len * p.n_heads);
  const int T = clamp_seq_len(p.seq_lens[b], p.q_len, p.max_seq_len, p.max_pages, p.status, false);
  const int ns = (T + kSplitTokens - 1) / kSplitTokens;
  __half *dst = p.out + static_cast<size_t>(row) * D + lane * PER;
  if (ns == 1) return;                       // the split kernel wrote this row
  float acc[PER];
#pragma unroll
  for (int e = 0; e < PER; ++e) acc[e] = 0.f;
  float L = 0.f;
  if (ns > 1) {
    const float *lse = p.lse_part + static_cast<size_t>(row) * p.nsplit_max;
    float M = -INFINITY;
    for (int s = lane; s < ns; s += 32) M = fmaxf(M, lse[s]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    if (M != -INFINITY) {
      const float *op = p.o_part + static_cast<size_t>(row) * p.nsplit_max * D + lane * PER;
      for (int s0 = 0; s0 < ns; s0 += 32) {
        const float w_l = (s0 + lane < ns) ? fast_exp2(lse[s0 + lane] - M) : 0.f;
        const int cnt = min(32, ns - s0);
        for (int j = 0; j < cnt; ++j) {
          const float w = __shfl_sync(0xffffffffu, w_l, j);
          L += w;
          const float4 *src = reinterpret_cast<const float4 *>(op + static_cast<size_t>(s0 + j) * D);
#pragma unroll
          for (int q4 = 0; q4 < PER / 4; ++q4) {
            const float4 x = src[q4];
            acc[4 * q4 + 0] = fmaf(w, x.x, acc[4 * q4 + 0]);
            acc[4 * q4 + 1] = fmaf(w, x.y, acc[4 * q4 + 1]);
            acc[4 * q4 + 2] = fmaf(w, x.z, acc[4 * q4 + 2]);
            acc[4 * q4 + 3] = fmaf(w, x.w, acc[4 * q4 + 3]);
          }
        }
      }
    }
  }
  const float inv = L > 0.f ? 1.f / L : 0.f;    // ns == 0 (empty sequence) writes zeros
#pragma unroll
  for (int q4 = 0; q4 < PER / 4; ++q4) {
    uint2 h;
    h.x = pack_half2(acc[4 * q4 + 0] * inv, acc[4 * q4 + 1] * inv);
    h.y = pack_half2(acc[4 * q4 + 2] * inv, acc[4 * q4 + 3] * inv);
    *reinterpret_cast<uint2 *>(dst + 4 * q4) = h;
  }
}

cudaError_t launch_combine(int D, const CombineParams &p, cudaStream_t st) {
  const unsigned grid = static_cast<unsigned>((p.rows + 3) / 4);
  if (D == 128)
    combine_kernel<128><<<grid, 128, 0, st>>>(p);
  else
    combine_kernel<256><<<grid, 128, 0, st>>>(p);
  return cudaGetLastError();
}

}  // namespace memra
