// K3: log-sum-exp combine of the split-K partials.
//
// For a query row whose visible keys (those up to its own position) span
// several splits, the split kernel left (o_s = O_s / l_s, lse_s = m_s + log2 l_s) per split.  The exact
// merge is  out = sum_s 2^(lse_s - M) o_s / sum_s 2^(lse_s - M),  M = max lse_s
// (splits with no visible key have lse = -inf and weight 0).  One CTA per
// row with up to 16 warps; warp w takes splits w, w+16, ... (eight in flight),
// each lane owning D/32 consecutive outputs, so every split's partial is one
// coalesced 512 B (D 128) or 1 KiB (D 256) read; the warps then reduce
// through shared memory.  Launched as a programmatic dependent of the split
// kernel, whose CTAs allow it as soon as they have started, so its launch
// overlaps the split kernel's work.
#include <cuda_runtime.h>

#include "decode_kernel.cuh"

namespace memra {

constexpr int kCombineMaxWarps = 16;

template <int D>
__global__ void __launch_bounds__(kCombineMaxWarps * 32) combine_kernel(const CombineParams p) {
  constexpr int PER = D / 32;                       // outputs per lane
  constexpr int BATCH = 8;                          // splits in flight per warp
  __shared__ float red[kCombineMaxWarps][D];
  __shared__ float redl[kCombineMaxWarps];
  __shared__ float mx[kCombineMaxWarps];
  const int row = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nw = blockDim.x >> 5;
  const int b = row / (p.q_len * p.n_heads);
  const int qi = (row / p.n_heads) % p.q_len;
  // Keys visible to this row's position (its own split plan, as in the split
  // kernel).  The lengths are read before the wait for the split kernel: they
  // were complete before that kernel started, and this grid launches only once
  // each of its CTAs has passed its own wait.
  const int Tseq = clamp_seq_len(p.seq_lens[b], p.q_len, p.max_seq_len, p.max_pages, p.ring, p.status, false);
  const int ns = key_range(Tseq, p.q_len, qi, p.window, 0, p.split_target).ns;
  grid_dependency_wait();                           // the split kernel's partials are complete
  __half *dst = p.out + static_cast<size_t>(row) * D;
  if (ns == 0) {                                    // no visible key: zeros
    for (int j = threadIdx.x; j < D; j += blockDim.x) dst[j] = __float2half(0.f);
    return;
  }
  if (ns == 1) return;                              // the split kernel wrote this row
  const float *lse = p.lse_part + static_cast<size_t>(row) * p.nsplit_max;
  const float *op = p.o_part + static_cast<size_t>(row) * p.nsplit_max * D + lane * PER;
  float acc[PER];
#pragma unroll
  for (int e = 0; e < PER; ++e) acc[e] = 0.f;
  float L = 0.f;
  // Warp w owns splits w, w + nw, ...; each batch issues all of its loads
  // (partials and their lse) before the block-wide maximum is known, so the
  // whole row costs one memory round trip per BATCH x nw splits.
  float M = -INFINITY;
  for (int base = 0; base < ns; base += BATCH * nw) {
    float4 x[BATCH][PER / 4];
    float ls[BATCH];
#pragma unroll
    for (int u = 0; u < BATCH; ++u) {
      const int sidx = base + warp + u * nw;
      const bool ok = sidx < ns;
      ls[u] = ok ? lse[sidx] : -INFINITY;
      const float4 *src = reinterpret_cast<const float4 *>(op + static_cast<size_t>(ok ? sidx : 0) * D);
#pragma unroll
      for (int q4 = 0; q4 < PER / 4; ++q4) x[u][q4] = ok ? src[q4] : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    // block-wide maximum of this batch's lse (and the previous batches')
    float m = M;
#pragma unroll
    for (int u = 0; u < BATCH; ++u) m = fmaxf(m, ls[u]);
    if (lane == 0) mx[warp] = m;
    __syncthreads();
    float mnew = mx[0];
    for (int w = 1; w < nw; ++w) mnew = fmaxf(mnew, mx[w]);
    __syncthreads();
    if (mnew != -INFINITY) {
      // rescale what was accumulated against the old maximum
      const float alpha = M == -INFINITY ? 0.f : fast_exp2(M - mnew);
      L *= alpha;
#pragma unroll
      for (int e = 0; e < PER; ++e) acc[e] *= alpha;
#pragma unroll
      for (int u = 0; u < BATCH; ++u) {
        const float wgt = ls[u] == -INFINITY ? 0.f : fast_exp2(ls[u] - mnew);
        L += wgt;
#pragma unroll
        for (int q4 = 0; q4 < PER / 4; ++q4) {
          acc[4 * q4 + 0] = fmaf(wgt, x[u][q4].x, acc[4 * q4 + 0]);
          acc[4 * q4 + 1] = fmaf(wgt, x[u][q4].y, acc[4 * q4 + 1]);
          acc[4 * q4 + 2] = fmaf(wgt, x[u][q4].z, acc[4 * q4 + 2]);
          acc[4 * q4 + 3] = fmaf(wgt, x[u][q4].w, acc[4 * q4 + 3]);
        }
      }
      M = mnew;
    }
  }
#pragma unroll
  for (int e = 0; e < PER; ++e) red[warp][lane * PER + e] = acc[e];
  if (lane == 0) redl[warp] = L;
  __syncthreads();
  for (int j = threadIdx.x; j < D / 2; j += blockDim.x) {
    float a0 = 0.f, a1 = 0.f, l = 0.f;
    for (int w = 0; w < nw; ++w) {
      a0 += red[w][2 * j];
      a1 += red[w][2 * j + 1];
      l += redl[w];
    }
    const float inv = l > 0.f ? 1.f / l : 0.f;
    reinterpret_cast<__half2 *>(dst)[j] = __floats2half2_rn(a0 * inv, a1 * inv);
  }
}

cudaError_t launch_combine(int D, const CombineParams &p, cudaStream_t st) {
  if (p.rows == 0) return cudaSuccess;
  int nw = p.nsplit_max < kCombineMaxWarps ? p.nsplit_max : kCombineMaxWarps;
  if (nw < 1) nw = 1;
  const dim3 grid(static_cast<unsigned>(p.rows)), block(static_cast<unsigned>(nw * 32));
  if (D == 128) return launch_pdl(combine_kernel<128>, grid, block, 0, st, p);
  return launch_pdl(combine_kernel<256>, grid, block, 0, st, p);
}

}  // namespace memra
