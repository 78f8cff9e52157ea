// Cascade decode: attention over a prefix that every sequence of the call
// shares, read and dequantized once per KV head for all of the call's query
// rows, on the fifth-generation tensor cores.
//
// memra serves many requests over one shared prefix (README introduction: the
// 4,860-token shared-prefix serving shape at concurrency 16; "Request reuse and
// admission").  Plain decode dequantizes each shared page once per sequence.
// Here the query rows of one KV head -- every sequence, query position and
// query head of its group, 128 to a tile -- are the M side of tcgen05 MMAs
// whose accumulators live in tensor memory: the one place on the decode path
// that is a dense contraction.  The attention is exact and comes in three
// launches merged by log-sum-exp:
//   * the prefix pass: CTA (run of 64-token chunks, KV head, row tile) stages
//     each chunk's prefix pages with bulk copies, dequantizes K and V once into
//     fp16 tiles in shared memory, computes S = Q K^T (M = 128 rows, N = chunk
//     tokens, K = head_dim) into tensor memory, keeps an online softmax per row
//     across its chunks, writes P in fp16 back to shared memory and
//     accumulates O += P V (N = head_dim, K = chunk tokens) in tensor memory.
//     At the end it writes one partial per row, (o = O / l, lse = m + log2 l),
//     the row by one bulk copy.  At head_dim 128 the pass is warp-specialized
//     (cascade_prefix_ws_kernel: staging, MMA and softmax warps, one thread
//     per row); at 256 its warps take the phases in turn (cascade_prefix_kernel,
//     two threads per row, one per column half);
//   * the split kernel over each sequence's own keys, from the prefix end on,
//     on the SMs the prefix pass leaves free;
//   * cascade_combine_kernel: the log-sum-exp merge of both, one CTA per row.
//
// Values enter the MMAs exactly, or nearly: fp8 and NVFP4 codes (times their
// e4m3 block scale) are exact in fp16, with the float32 tensor scale applied to
// the fp32 scores or output; a q8_0 / q5_1 / q4_0 value is staged at half its
// size as an fp16 pair hi + lo (the rounded product and its residual from one
// FMA; for q5_1 also a TwoSum with m/2), both parts enter the same accumulator,
// and the factor 2 returns in fp32.  The pair is exact for q8_0 and q4_0 while
// the residual is representable: its last bit is ulp(d)/2 (halved value), so
// exact for d >= 2^-13; for smaller d the residual is rounded to an fp16
// subnormal, off by at most 2^-25 (2^-24 on the value).  q5_1's d q + m is
// within ~2^-22 of the block's scale, and also within 2^-24 absolute when m/2
// or the residual falls below the fp16 subnormal step.  Halving keeps every value of an fp16-range block
// finite.  A row's bytes depend on its own query and the keys only (no value of
// one row enters another's), and on the prefix length, which fixes the chunks.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <type_traits>

#include "cascade.cuh"
#include "decode_kernel.cuh"
#include "tcgen05.cuh"

namespace memra {
namespace {

constexpr int kThreads = 256;         // 8 warps: two per tensor-memory lane quarter
constexpr int kTileRows = 128;
constexpr uint32_t kSmemLimit = 232448;

__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}

__device__ __forceinline__ uint32_t lds16(uint32_t addr) {
  unsigned short v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr));
  return v;
}

__device__ __forceinline__ uint32_t lds8(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.u8 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}

// One thread: copy `bytes` (a multiple of 16, both addresses 16-byte aligned)
// from shared to global memory through the async proxy, as one bulk
// async-group of this thread.
__device__ __forceinline__ void bulk_store_s2g(void *dst, uint32_t src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(src), "r"(bytes)
               : "memory");
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// One thread: its bulk stores have completed, writes performed (before the
// CTA, and its shared memory, goes away).
__device__ __forceinline__ void bulk_store_wait() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Global row id of row r of a KV head's row tiles: sequence b = r / (q_len *
// group), then query position and head of the group.
__device__ __forceinline__ size_t prefix_row_id(const CascadeParams &p, int kvh, int r) {
  const int rows_per_seq = p.q_len * p.group;
  const int b = r / rows_per_seq, rem = r % rows_per_seq;
  return (static_cast<size_t>(b) * p.q_len + rem / p.group) * p.n_heads + kvh * p.group + rem % p.group;
}

__device__ __forceinline__ void sts128(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}

__device__ __forceinline__ uint32_t h2_bits(__half2 h) { return *reinterpret_cast<uint32_t *>(&h); }
__device__ __forceinline__ __half2 bits_h2(uint32_t u) { return *reinterpret_cast<__half2 *>(&u); }

// fp16 of the low e4m3 byte of `byte`, broadcast to both halves.
__device__ __forceinline__ __half2 e4m3_scale_h2(uint32_t byte) {
  const uint32_t h = e4m3x2_to_half2(byte & 0xFFu) & 0xFFFFu;
  return bits_h2(h | (h << 16));
}

// Raw shared-memory words of one K staging item (token t of a staged page,
// dims 8u .. 8u + 7): the 8 code bytes (NVFP4: the 8-byte group holding the
// item's 16 nibbles) and the block-scale bits.  Layout formulas of memra.h.
struct KRaw {
  uint2 w;
  uint32_t s;
};

template <int D, int KF>
__device__ __forceinline__ KRaw load_k8(uint32_t seg, int t, int u) {
  constexpr int NB = D / 32;
  const int b = u >> 2, c = u & 3;
  const uint32_t lane = 4 * (t & 7) + c;
  KRaw r;
  if constexpr (KF == MEMRA_KV_NVFP4) {
    r.w = lds64(seg + ((b >> 1) * 32 + lane) * 16 + (b & 1) * 8);
    r.s = lds8(seg + 8 * D + t * (D / 16) + (u >> 1));
  } else {
    r.w = lds64(seg + (((t >> 3) * (NB / 2) + (b >> 1)) * 32 + lane) * 16 + (b & 1) * 8);
    r.s = KF == MEMRA_KV_Q8_0 ? lds16(seg + 16 * D + (t * NB + b) * 2) : 0u;
  }
  return r;
}

// The item's 8 values as fp16 (hi) plus, for q8_0, the low parts (lo).
template <int KF>
__device__ __forceinline__ void convert_k8(const KRaw &r, int t, uint32_t (&hi)[4], uint32_t (&lo)[4]) {
  if constexpr (KF == MEMRA_KV_Q8_0) {
    const __half2 d2 = bits_h2(r.s | (r.s << 16));
    const __half2 half = __float2half2_rn(0.5f), off = __float2half2_rn(-576.f);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      // codes are stored as q + 128: splice under 1024 -> 1152 + q, then q / 2 exactly
      const uint32_t word = k < 2 ? r.w.x : r.w.y;
      const __half2 code = bits_h2(__byte_perm(word, 0x64646464u, k & 1 ? 0x4342 : 0x4140));
      const __half2 qh = __hfma2(code, half, off);
      const __half2 h = __hmul2(qh, d2);
      hi[k] = h2_bits(h);
      lo[k] = h2_bits(__hfma2(qh, d2, __hneg2(h)));
    }
  } else if constexpr (KF == MEMRA_KV_FP8_E4M3) {
    e4m3x4_to_half2x2(r.w.x, hi[0], hi[1]);
    e4m3x4_to_half2x2(r.w.y, hi[2], hi[3]);
  } else {   // NVFP4: bytes t/8 and t/8 + 2 of each word hold the (2k, 2k + 1) dim pairs
    const int sh = 8 * (t >> 3);
    const __half2 s2 = e4m3_scale_h2(r.s);
    hi[0] = h2_bits(__hmul2(bits_h2(e2m1x2_to_half2((r.w.x >> sh) & 0xFFu)), s2));
    hi[1] = h2_bits(__hmul2(bits_h2(e2m1x2_to_half2((r.w.x >> (sh + 16)) & 0xFFu)), s2));
    hi[2] = h2_bits(__hmul2(bits_h2(e2m1x2_to_half2((r.w.y >> sh) & 0xFFu)), s2));
    hi[3] = h2_bits(__hmul2(bits_h2(e2m1x2_to_half2((r.w.y >> (sh + 16)) & 0xFFu)), s2));
  }
}

// Raw words of one V staging task of the q5_1 / q4_0 / fp8 layouts: page half
// ph, block b, dim group vg and pair h (dims 32 b + 4 vg + 2 h, + 1), tokens
// 8 ph + 2 c + f.
struct VRaw {
  uint32_t lw[4];              // per c: the code word of pair h
  uint32_t hw[4], dw[4], mw[4];
};

template <int D, int VF>
__device__ __forceinline__ VRaw load_v_task(uint32_t seg, int ph, int b, int vg, int h) {
  constexpr int NB = D / 32;
  VRaw r;
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const uint32_t lane = 4 * vg + c;
    r.hw[c] = r.dw[c] = r.mw[c] = 0u;
    if constexpr (VF == MEMRA_KV_FP8_E4M3) {
      r.lw[c] = lds32(seg + (b * 32 + lane) * 16 + 8 * h + 4 * ph);
    } else {
      const uint32_t doff = ((c * NB + b) * 4 + 2 * ph) * 2;
      r.lw[c] = lds32(seg + ((b >> 1) * 32 + lane) * 16 + (b & 1) * 8 + 4 * h);
      if constexpr (VF == MEMRA_KV_Q5_1) {
        r.hw[c] = lds32(seg + 8 * D + (lane * (NB / 2) + (b >> 1)) * 4);
        r.dw[c] = lds32(seg + 10 * D + doff);
        r.mw[c] = lds32(seg + 11 * D + doff);
      } else {
        r.dw[c] = lds32(seg + 8 * D + doff);
      }
    }
  }
  return r;
}

// The task's values: for dim s of the pair, tokens 2c, 2c + 1 as one fp16
// pair hi[s][c] (and lo[s][c] for q5_1 / q4_0).
template <int VF>
__device__ __forceinline__ void convert_v_task(const VRaw &r, int ph, int b, int h, uint32_t (&hi)[2][4],
                                               uint32_t (&lo)[2][4]) {
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    if constexpr (VF == MEMRA_KV_FP8_E4M3) {
      // bytes 2 s + f of the word: (s = 0: f = 0, 1), (s = 1: f = 0, 1)
      e4m3x4_to_half2x2(r.lw[c], hi[0][c], hi[1][c]);
    } else {
      // Both tokens of the pair (f = 0, 1) at once: their codes sit 16 bits
      // apart in the words, and their scales are the two halves of dw, mw.
      // The value, halved, is d q/2 (+ m/2 for q5_1) as hi + lo fp16 parts:
      // the product rounded and its residual (one FMA), and for q5_1 the
      // rounded sum with m/2 and its error (TwoSum).  The _rn operations are
      // never contracted into FMAs.  The parts are exact while the residual
      // is representable in fp16 (d >= 2^-13); below that, the residual and
      // m/2 are rounded to fp16 subnormals (at most 2^-25 off each).
      const __half2 d2 = bits_h2(r.dw[c]);
#pragma unroll
      for (int s = 0; s < 2; ++s) {
        const int sh = 8 * ph + 4 * s;
        uint32_t codes = (r.lw[c] >> sh) & 0x000F000Fu;
        if constexpr (VF == MEMRA_KV_Q5_1) codes |= ((r.hw[c] >> (sh + 2 * (b & 1) + h)) & 0x00010001u) << 4;
        // 1024 + q as fp16, then q/2 (q5_1) or (q - 8)/2 (q4_0), exactly
        const __half2 q2 = __hfma2(bits_h2(codes | 0x64006400u), __float2half2_rn(0.5f),
                                   __float2half2_rn(VF == MEMRA_KV_Q5_1 ? -512.f : -516.f));
        const __half2 p_hi = __hmul2_rn(q2, d2);
        const __half2 p_lo = __hfma2(q2, d2, __hneg2(p_hi));
        if constexpr (VF == MEMRA_KV_Q5_1) {
          const __half2 m2 = __hmul2_rn(bits_h2(r.mw[c]), __float2half2_rn(0.5f));
          const __half2 s2 = __hadd2_rn(p_hi, m2);
          const __half2 bb = __hsub2_rn(s2, p_hi);
          const __half2 e2 = __hadd2_rn(__hsub2_rn(p_hi, __hsub2_rn(s2, bb)), __hsub2_rn(m2, bb));
          hi[s][c] = h2_bits(s2);
          lo[s][c] = h2_bits(__hadd2_rn(e2, p_lo));
        } else {
          hi[s][c] = h2_bits(p_hi);
          lo[s][c] = h2_bits(p_lo);
        }
      }
    }
  }
}

template <int D, int KF, int VF>
__global__ void __launch_bounds__(kThreads, cascade_ctas_per_sm(D)) cascade_prefix_kernel(const CascadeParams p) {
  constexpr int NC = cascade_chunk_tokens(D);       // prefix tokens of one chunk
  constexpr int H = NC / 2;                         // tokens staged at a time (one half)
  constexpr int NPG = NC / kPage;
  constexpr int HPG = H / kPage;                    // pages of a half
  constexpr int NB = D / 32;
  constexpr int KSEG = k_seg_bytes(KF, D);
  constexpr int VSEG = v_seg_bytes(VF, D);
  constexpr bool kKLo = KF == MEMRA_KV_Q8_0;
  constexpr bool kVLo = VF == MEMRA_KV_Q5_1 || VF == MEMRA_KV_Q4_0;
  constexpr float kLazy = 8.f;                      // log2 units: P stays <= 256 between rescales
  // Shared memory (byte offsets): the Q tile; one half of K^ (hi, lo; token
  // rows) and P after the scores; one half of V^T (hi, lo; dim rows); two
  // buffers of raw pages (a chunk's K pages, then its V pages), the next
  // chunk's copies landing in one while the other is staged; the softmax
  // exchange; the page ids of the CTA's chunks; barriers.  The output rows
  // reuse Q, K^, V^T and the raw buffers once O is done.
  constexpr uint32_t QB = kTileRows * D * 2, KHB = H * D * 2, VHB = D * H * 2;
  constexpr uint32_t RAWB = NPG * (KSEG + VSEG);
  constexpr uint32_t OFF_Q = 0, OFF_K = QB, OFF_V = OFF_K + 2 * KHB, OFF_RAW = OFF_V + 2 * VHB;
  constexpr uint32_t ROWB = D * 4 + 16;                       // padded output row in shared memory
  constexpr uint32_t TCOLS = cascade_tmem_cols(D);            // O at column 0, S at column D
  // one raw buffer when the CTA has one chunk, two when it loops over several
  const uint32_t nbuf = p.cpc > 1 ? 2u : 1u;
  const uint32_t OFF_X = OFF_RAW + nbuf * RAWB, OFF_PID = OFF_X + 4 * kTileRows * 4,
                 OFF_BAR = OFF_PID + 4 * NPG * p.cpc;
  static_assert(OFF_RAW + 2 * RAWB + 4 * kTileRows * 4 + 4 * NPG * kCascadeMaxChunksPerCta + 64 ==
                    cascade_smem_plan(D, KSEG, VSEG, kCascadeMaxChunksPerCta) &&
                    OFF_RAW + RAWB + 4 * kTileRows * 4 + 4 * NPG + 64 == cascade_smem_plan(D, KSEG, VSEG, 1),
                "shared-memory plan");
  static_assert(cascade_smem_bytes(D, KSEG, VSEG, kCascadeMaxChunksPerCta) <= kSmemLimit, "shared memory");
  static_assert(kTileRows * ROWB <= OFF_RAW + RAWB, "output rows below the exchange");
  static_assert(kTileRows * NC * 2 <= 2 * KHB, "P fits the K^ half");
  static_assert(D + NC <= static_cast<int>(TCOLS), "O and S fit the tensor memory");
  static_assert(KSEG % 16 == 0 && VSEG % 16 == 0 && OFF_RAW % 16 == 0 && RAWB % 16 == 0 && (4 * NPG) % 16 == 0,
                "alignment");
  constexpr int QIT = kTileRows * (D / 8) / kThreads;        // Q items per thread
  constexpr int KIT = H * (D / 8) / kThreads;                // K items per thread and half
  constexpr int VTASKS = VF == MEMRA_KV_NVFP4 ? HPG * 2 * (D / 16) * 8 : HPG * 2 * NB * 8 * 2;
  constexpr int VIT = (VTASKS + kThreads - 1) / kThreads;    // V tasks per thread and half
  static_assert(QIT * kThreads == kTileRows * (D / 8) && KIT * kThreads == H * (D / 8), "whole items");
  static_assert(VIT * kThreads == VTASKS || (VIT == 1 && VTASKS % 32 == 0), "whole warps of tasks");

  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sb = smem_addr(smem);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t bar_raw0 = sb + OFF_BAR, bar_s = bar_raw0 + 16, bar_o = bar_raw0 + 24;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + OFF_BAR + 32);
  int *pid_s = reinterpret_cast<int *>(smem + OFF_PID);        // [chunk of the CTA][page], -1 = none
  float *xm = reinterpret_cast<float *>(smem + OFF_X);
  float *xl = xm + 2 * kTileRows;

  const int kvh = blockIdx.y;
  const int rows = p.batch * p.q_len * p.group;                  // query rows of one KV head
  const int r0 = blockIdx.z * kTileRows;
  const int c0 = blockIdx.x * p.cpc;                             // this CTA's chunks: c0 .. c0 + nck - 1
  const int nck = max(0, min(p.cpc, p.n_chunks - c0));
  const int rows_per_seq = p.q_len * p.group;

  if (warp == 0) {
    tc::tmem_alloc(smem_addr(tmem_slot), TCOLS);
    tc::tmem_relinquish();
  }
  if (tid == 32) {
    mbar_init(bar_raw0, 1);
    mbar_init(bar_raw0 + 8, 1);
    mbar_init(bar_s, 1);
    mbar_init(bar_o, 1);
    fence_barrier_init();
  }
  grid_dependency_wait();          // q, the pools and the tables are written
  allow_dependent_launch();        // the own-key split kernel may start beside this one

  // Page ids of all of this CTA's chunks, from the first sequence's table.
  for (int i = tid; i < nck * NPG; i += kThreads) {
    const int tok = c0 * NC + i * kPage;
    int pid = -1;
    if (tok < p.prefix_len) {
      pid = p.page_table[tok / kPage];
      if (pid < 0 || pid >= p.num_pages) {
        flag_error(p.status, MEMRA_DEVERR_BAD_PAGE);
        pid = -1;
      }
    }
    pid_s[i] = pid;
  }

  // Q rows of the tile in core-matrix order: item i = (row group, 8-dim group,
  // row in group), shared-memory byte 16 i.  All of a thread's loads are in
  // flight together, beside the page-id loads.
  uint4 qv[QIT];
#pragma unroll
  for (int it = 0; it < QIT; ++it) {
    const int i = tid + it * kThreads;
    const int rest = i >> 3, u = rest % (D / 8);
    const int r = r0 + (rest / (D / 8)) * 8 + (i & 7);
    qv[it] = make_uint4(0, 0, 0, 0);
    if (r < rows) {
      const int b = r / rows_per_seq, rem = r % rows_per_seq;
      const size_t rowid = (static_cast<size_t>(b) * p.q_len + rem / p.group) * p.n_heads + kvh * p.group +
                           rem % p.group;
      qv[it] = *reinterpret_cast<const uint4 *>(p.q + rowid * D + 8 * u);
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  // Copies of chunk ci (of this CTA) into raw buffer ci % 2: one bulk copy per
  // page for K and for V, or a plain arrival when the chunk has no page.
  const size_t kstride = static_cast<size_t>(p.n_kv_heads) * KSEG, vstride = static_cast<size_t>(p.n_kv_heads) * VSEG;
  auto issue = [&](int ci) {
    const uint32_t buf = sb + OFF_RAW + (ci & 1) * RAWB, bar = bar_raw0 + 8 * (ci & 1);
    uint32_t bytes = 0;
    for (int i = 0; i < NPG; ++i) bytes += pid_s[ci * NPG + i] >= 0 ? KSEG + VSEG : 0;
    if (!bytes) {
      mbar_arrive(bar);
      return;
    }
    mbar_arrive_expect_tx(bar, bytes);
    for (int i = 0; i < NPG; ++i) {
      const int pg = pid_s[ci * NPG + i];
      if (pg < 0) continue;
      bulk_copy_g2s_nohint(buf + i * KSEG, p.k_pool + pg * kstride + static_cast<size_t>(kvh) * KSEG, KSEG, bar);
      bulk_copy_g2s_nohint(buf + NPG * KSEG + i * VSEG, p.v_pool + pg * vstride + static_cast<size_t>(kvh) * VSEG,
                           VSEG, bar);
    }
  };
  if (tid == 0) {
    if (nck > 0) issue(0);
    if (nck > 1) issue(1);
  }
  int issued = min(nck, 2), consumed = 0;    // chunks whose copies were issued / waited for (all threads)
#pragma unroll
  for (int it = 0; it < QIT; ++it) sts128(sb + OFF_Q + 16 * (tid + it * kThreads), qv[it]);

  bool ok = true;
  uint32_t pmask = 0;              // pages of the current chunk that hold keys, one bit each
  uint32_t rawk = 0, rawv = 0;     // the current chunk's raw K and V pages

  // K^ of half hf (token rows, dims along K) at the K buffer: item i =
  // (token group, 8-dim group, token in group) at byte 16 i of hi and lo.
  auto stage_k = [&](int hf) {
    KRaw kr[KIT];
#pragma unroll
    for (int it = 0; it < KIT; ++it) {
      const int i = tid + it * kThreads;
      const int n = hf * H + ((i >> 3) / (D / 8)) * 8 + (i & 7);
      kr[it] = load_k8<D, KF>(rawk + (n / kPage) * KSEG, n % kPage, (i >> 3) % (D / 8));
    }
#pragma unroll
    for (int it = 0; it < KIT; ++it) {
      const int i = tid + it * kThreads;
      const int n = hf * H + ((i >> 3) / (D / 8)) * 8 + (i & 7);
      uint32_t hi[4] = {0, 0, 0, 0}, lo[4] = {0, 0, 0, 0};
      if (ok && ((pmask >> (n / kPage)) & 1u)) convert_k8<KF>(kr[it], n % kPage, hi, lo);
      sts128(sb + OFF_K + 16 * i, make_uint4(hi[0], hi[1], hi[2], hi[3]));
      if constexpr (kKLo) sts128(sb + OFF_K + KHB + 16 * i, make_uint4(lo[0], lo[1], lo[2], lo[3]));
    }
  };
  // V^T of half hf (dim rows, tokens along K) at the V buffer: a task is one
  // staged page half (8 tokens) and a group of dims; it writes one 16-byte row
  // of a core matrix per dim: dim dd, token group g at ((dd/8) * H/8 + g) * 128 + (dd%8) * 16.
  auto vt_store = [&](int dd, int g, uint4 h, uint4 l) {
    const uint32_t off = ((dd >> 3) * (H / 8) + g) * 128 + (dd & 7) * 16;
    sts128(sb + OFF_V + off, h);
    if constexpr (kVLo) sts128(sb + OFF_V + VHB + off, l);
  };
  auto stage_v = [&](int hf) {
    if constexpr (VF == MEMRA_KV_NVFP4) {
      // task (page, half page, 16-dim block b16, rr): dims 16 b16 + rr and + 8
      uint32_t cw[VIT][4], sw[VIT][4];
#pragma unroll
      for (int it = 0; it < VIT; ++it) {
        const int task = tid + it * kThreads;
        if (task >= VTASKS) break;
        const int rr = task & 7, b16 = (task >> 3) % (D / 16), ps = hf * HPG + task / (16 * (D / 16));
        const uint32_t seg = rawv + ps * VSEG;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          cw[it][c] = lds32(seg + ((b16 >> 2) * 32 + 4 * rr + c) * 16 + (b16 & 3) * 4);
          sw[it][c] = lds32(seg + 8 * D + (c * (D / 16) + b16) * 4);
        }
      }
#pragma unroll
      for (int it = 0; it < VIT; ++it) {
        const int task = tid + it * kThreads;
        if (task >= VTASKS) break;
        const int rr = task & 7, b16 = (task >> 3) % (D / 16), ph = (task / (8 * (D / 16))) & 1,
                  psl = task / (16 * (D / 16));
        uint32_t h0[4] = {0, 0, 0, 0}, h1[4] = {0, 0, 0, 0};
        if (ok && ((pmask >> (hf * HPG + psl)) & 1u)) {
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            __half2 v[2];
#pragma unroll
            for (int f = 0; f < 2; ++f) {
              const int sh = 8 * (f + 2 * ph);
              v[f] = __hmul2(bits_h2(e2m1x2_to_half2((cw[it][c] >> sh) & 0xFFu)), e4m3_scale_h2(sw[it][c] >> sh));
            }
            h0[c] = h2_bits(__lows2half2(v[0], v[1]));
            h1[c] = h2_bits(__highs2half2(v[0], v[1]));
          }
        }
        const uint4 z = make_uint4(0, 0, 0, 0);
        vt_store(16 * b16 + rr, 2 * psl + ph, make_uint4(h0[0], h0[1], h0[2], h0[3]), z);
        vt_store(16 * b16 + rr + 8, 2 * psl + ph, make_uint4(h1[0], h1[1], h1[2], h1[3]), z);
      }
    } else {
      // task (page, half page, block b, vg, pair h): dims 32 b + 4 vg + 2 h + s, tokens 8 half + 2 c + f
      VRaw vr[VIT];
#pragma unroll
      for (int it = 0; it < VIT; ++it) {
        const int task = tid + it * kThreads;
        if (task >= VTASKS) break;
        const int h = task & 1, vg = (task >> 1) & 7, b = (task >> 4) % NB, ph = (task / (16 * NB)) & 1,
                  ps = hf * HPG + task / (32 * NB);
        vr[it] = load_v_task<D, VF>(rawv + ps * VSEG, ph, b, vg, h);
      }
#pragma unroll
      for (int it = 0; it < VIT; ++it) {
        const int task = tid + it * kThreads;
        if (task >= VTASKS) break;
        const int h = task & 1, vg = (task >> 1) & 7, b = (task >> 4) % NB, ph = (task / (16 * NB)) & 1,
                  psl = task / (32 * NB);
        uint32_t hi[2][4], lo[2][4];
        convert_v_task<VF>(vr[it], ph, b, h, hi, lo);
        const bool have = ok && ((pmask >> (hf * HPG + psl)) & 1u);
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const uint4 hv = have ? make_uint4(hi[e][0], hi[e][1], hi[e][2], hi[e][3]) : make_uint4(0, 0, 0, 0);
          const uint4 lv = have && kVLo ? make_uint4(lo[e][0], lo[e][1], lo[e][2], lo[e][3]) : make_uint4(0, 0, 0, 0);
          vt_store(32 * b + 4 * vg + 2 * h + e, 2 * psl + ph, hv, lv);
        }
      }
    }
  };
  // S[:, half hf] = Q K^T (N = H tokens, K = head_dim in steps of 16) into
  // tensor-memory columns D + hf * H ..
  constexpr uint32_t idesc_s = tc::idesc_f16_f32(kTileRows, H);
  constexpr uint32_t idesc_o = tc::idesc_f16_f32(kTileRows, D);
  auto mma_s = [&](int hf) {
    tc::fence_after_sync();
#pragma unroll 1
    for (int ks = 0; ks < D / 16; ++ks) {
      const uint64_t a = tc::smem_desc(sb + OFF_Q + 256 * ks, 128, (D / 8) * 128);
      tc::mma_f16(tmem + D + hf * H, a, tc::smem_desc(sb + OFF_K + 256 * ks, 128, (D / 8) * 128), idesc_s, ks > 0);
      if constexpr (kKLo)
        tc::mma_f16(tmem + D + hf * H, a, tc::smem_desc(sb + OFF_K + KHB + 256 * ks, 128, (D / 8) * 128), idesc_s,
                    1);
    }
    tc::commit(bar_s);
  };
  // O (+)= P[:, half hf] V^T (K = the half's tokens in steps of 16); the first
  // MMA of the CTA's first chunk starts the accumulator
  auto mma_o = [&](int hf, bool first_chunk) {
    tc::fence_after_sync();
#pragma unroll 1
    for (int ks = 0; ks < H / 16; ++ks) {
      const uint64_t a = tc::smem_desc(sb + OFF_K + 256 * (hf * (H / 16) + ks), 128, (NC / 8) * 128);
      tc::mma_f16(tmem, a, tc::smem_desc(sb + OFF_V + 256 * ks, 128, (H / 8) * 128), idesc_o,
                  !first_chunk || hf > 0 || ks > 0);
      if constexpr (kVLo)
        tc::mma_f16(tmem, a, tc::smem_desc(sb + OFF_V + VHB + 256 * ks, 128, (H / 8) * 128), idesc_o, 1);
    }
    tc::commit(bar_o);
  };
  auto sync_tiles = [&]() {        // thread-written tiles -> the tensor cores (uniform result)
    fence_proxy_async();
    tc::fence_before_sync();
    ok = !__syncthreads_or(!ok);
  };

  // Online softmax over the CTA's chunks: thread (lane quarter, column half)
  // owns row rl and half colh of the chunk's columns and of O's.  The row's
  // reference maximum m moves only when a chunk's maximum passes it by more
  // than kLazy; then O (in tensor memory) and l are rescaled.  Both threads of
  // a row see the same maxima, so they take the same decisions.
  const int quarter = warp & 3, colh = warp >> 2;
  const int rl = quarter * 32 + lane;
  const uint32_t tlane = static_cast<uint32_t>(quarter * 32) << 16;
  constexpr int HC = NC / 2;
  float m_row = -INFINITY, l_row = 0.f;

#pragma unroll 1
  for (int ci = 0; ci < nck && ok; ++ci) {
    const int b = ci & 1;
    rawk = sb + OFF_RAW + b * RAWB;
    rawv = rawk + NPG * KSEG;
    pmask = 0;
#pragma unroll
    for (int i = 0; i < NPG; ++i) pmask |= (pid_s[ci * NPG + i] >= 0 ? 1u : 0u) << i;
    ok = mbar_wait_bounded(bar_raw0 + 8 * b, (ci >> 1) & 1, p.status);

    // first half of K, its scores; the first half of V meanwhile
    stage_k(0);
    sync_tiles();
    if (ok) consumed = ci + 1;
    if (ok && tid == 0) mma_s(0);
    stage_v(0);
    // second half of K once the first half's MMAs have read the buffer
    if (ok) ok = mbar_wait_bounded(bar_s, 0, p.status);
    stage_k(1);
    sync_tiles();
    if (ok && tid == 0) mma_s(1);
    if (ok) ok = mbar_wait_bounded(bar_s, 1, p.status);
    ok = !__syncthreads_or(!ok);
    if (!ok) break;

    tc::fence_after_sync();
    uint32_t sr[HC];
#pragma unroll
    for (int k0 = 0; k0 < HC; k0 += 16) tc::ld_32x32b_x16(tmem + tlane + D + colh * HC + k0, sr + k0);
#pragma unroll
    for (int k0 = 0; k0 < HC; k0 += 16) tc::wait_ld(sr + k0);
    float mloc = -INFINITY;
#pragma unroll
    for (int k = 0; k < HC; ++k) {
      const bool valid = (pmask >> (colh * (HC / kPage) + k / kPage)) & 1u;
      const float v = valid ? __uint_as_float(sr[k]) * p.scale_log2 : -INFINITY;
      sr[k] = __float_as_uint(v);
      mloc = fmaxf(mloc, v);
    }
    xm[colh * kTileRows + rl] = mloc;
    __syncthreads();
    const float m_chunk = fmaxf(xm[rl], xm[kTileRows + rl]);
    float alpha = 1.f;
    if (m_chunk > m_row + kLazy) {           // also the first chunk with a key (m_row = -inf)
      if (m_row != -INFINITY) alpha = fast_exp2(m_row - m_chunk);
      m_row = m_chunk;
    }
    if (ci > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
      // O's rows of this warp (its column half) times alpha; 1 for the rows that keep their maximum
#pragma unroll 1
      for (int k0 = 0; k0 < D / 2; k0 += 16) {
        uint32_t orr[16];
        tc::ld_32x32b_x16(tmem + tlane + colh * (D / 2) + k0, orr);
        tc::wait_ld(orr);
#pragma unroll
        for (int e = 0; e < 16; ++e) orr[e] = __float_as_uint(__uint_as_float(orr[e]) * alpha);
        tc::st_32x32b_x16(tmem + tlane + colh * (D / 2) + k0, orr);
      }
      tc::wait_st();
    }
    // P (fp16) over the K buffer: row rl, token group g at ((rl/8) * NC/8 + g) * 128 + (rl%8) * 16
    float lsum = 0.f;
#pragma unroll
    for (int g = 0; g < HC / 8; ++g) {
      uint32_t w4[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float p0 = m_row == -INFINITY ? 0.f : fast_exp2(__uint_as_float(sr[8 * g + 2 * e]) - m_row);
        const float p1 = m_row == -INFINITY ? 0.f : fast_exp2(__uint_as_float(sr[8 * g + 2 * e + 1]) - m_row);
        const __half2 ph2 = __floats2half2_rn(p0, p1);
        const float2 back = __half22float2(ph2);
        lsum += back.x + back.y;
        w4[e] = h2_bits(ph2);
      }
      const int gg = colh * (HC / 8) + g;
      sts128(sb + OFF_K + ((rl >> 3) * (NC / 8) + gg) * 128 + (rl & 7) * 16, make_uint4(w4[0], w4[1], w4[2], w4[3]));
    }
    xl[colh * kTileRows + rl] = lsum;
    sync_tiles();
    l_row = l_row * alpha + (xl[rl] + xl[kTileRows + rl]);
    if (ok && tid == 0) mma_o(0, ci == 0);
    // second half of V once the first half's MMAs have read the buffer
    if (ok) ok = mbar_wait_bounded(bar_o, 0, p.status);
    stage_v(1);
    sync_tiles();                  // also: this chunk's raw pages are no longer read
    if (ok && tid == 0) {
      mma_o(1, ci == 0);
      if (ci + 2 < nck) issue(ci + 2);
    }
    if (ok) issued = min(nck, ci + 3);
    if (ok) ok = mbar_wait_bounded(bar_o, 1, p.status);
    ok = !__syncthreads_or(!ok);
  }

  if (ok && nck > 0) {
    tc::fence_after_sync();
    // o = O * v_post / l into padded shared-memory rows (Q, K^, P, V^T and the
    // raw buffers are no longer read); a row without keys writes zeros
    const float inv = l_row > 0.f ? p.v_post / l_row : 0.f;
#pragma unroll 1
    for (int k0 = 0; k0 < D / 2; k0 += 32) {
      uint32_t orr[32];
      tc::ld_32x32b_x16(tmem + tlane + colh * (D / 2) + k0, orr);
      tc::ld_32x32b_x16(tmem + tlane + colh * (D / 2) + k0 + 16, orr + 16);
      tc::wait_ld(orr);
      tc::wait_ld(orr + 16);
#pragma unroll
      for (int e = 0; e < 32; e += 4)
        sts128(sb + OFF_Q + rl * ROWB + (colh * (D / 2) + k0 + e) * 4,
               l_row > 0.f ? make_uint4(__float_as_uint(__uint_as_float(orr[e]) * inv),
                                        __float_as_uint(__uint_as_float(orr[e + 1]) * inv),
                                        __float_as_uint(__uint_as_float(orr[e + 2]) * inv),
                                        __float_as_uint(__uint_as_float(orr[e + 3]) * inv))
                           : make_uint4(0, 0, 0, 0));
    }
  }
  // This CTA's partial of each row: the row by one bulk copy of its padded
  // shared-memory row (both column halves, ordered for the async proxy by the
  // fence and the barrier), the lse by a plain store.  A row without keys, or
  // every row after a wait that gave up, gets lse = -inf, which the merge
  // never weighs.
  fence_proxy_async();
  __syncthreads();
  if (colh == 0 && r0 + rl < rows) {
    const size_t slot = prefix_row_id(p, kvh, r0 + rl) * p.n_parts + blockIdx.x;
    if (ok && nck > 0) bulk_store_s2g(p.o_pre + slot * D, sb + OFF_Q + rl * ROWB, D * 4);
    p.lse_pre[slot] = ok && nck > 0 && l_row > 0.f ? m_row + __log2f(l_row) : -INFINITY;
  }

  // Every sequence of the row tile must hold the same prefix pages and see all
  // of the prefix (flags only, off the critical path; one KV head checks).
  if (kvh == 0) {
    const int b_first = r0 / rows_per_seq, b_last = (min(rows, r0 + kTileRows) - 1) / rows_per_seq;
    const int pages = nck * NPG;
    for (int i = tid; i < (b_last - b_first + 1) * pages; i += kThreads) {
      const int bb = b_first + i / pages, j = c0 * NPG + i % pages;
      if (j * kPage < p.prefix_len && p.page_table[static_cast<size_t>(bb) * p.max_pages + j] != p.page_table[j])
        flag_error(p.status, MEMRA_DEVERR_PREFIX);
    }
    if (blockIdx.x == 0)
      for (int bb = b_first + tid; bb <= b_last; bb += kThreads)
        if (p.seq_lens[bb] - p.q_len < p.prefix_len) flag_error(p.status, MEMRA_DEVERR_BAD_SEQ_LEN);
  }
  // After a wait that gave up, the copies still in flight land (bounded) before the CTA leaves.
  if (!ok)
    for (int ci = consumed; ci < issued; ++ci) mbar_wait_bounded(bar_raw0 + 8 * (ci & 1), (ci >> 1) & 1, p.status);
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tmem, TCOLS);
  bulk_store_wait();               // the row copies this thread issued (none: returns at once)
}

// Warps of the warp-specialized pass: 4 softmax, kStageWarps staging, 1 MMA.
constexpr int kStageWarps = 8;
constexpr int kStageThreads = 32 * kStageWarps;
constexpr int kMmaWarp = 4 + kStageWarps;
constexpr int kWsThreads = 32 * (kMmaWarp + 1);

// Staging warps of the warp-specialized pass (named barrier 1): a barrier that
// also ANDs `ok` over them, so that they all take the same branch.
__device__ __forceinline__ bool staging_all(bool ok) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\tbar.red.and.pred q, 1, %2, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(ok ? 1u : 0u), "n"(kStageThreads)
      : "memory");
  return r != 0;
}

// The head_dim 128 prefix pass, warp-specialized: the three kinds of work of a
// chunk (dequantizing K and V into tensor-core tiles, the MMAs, the online
// softmax) run in separate warps and overlap across chunks through
// double-buffered tiles handed over by mbarriers.
//   * warps 0-3 (softmax): thread = query row; per chunk it reads the row's
//     scores from tensor memory, keeps the row's reference maximum (moved only
//     when a chunk passes it by more than kLazy, in log2 units), rescales O in
//     tensor memory when it moves, writes P (fp16) for the output MMA, and at
//     the end normalizes O;
//   * warps 4 .. 4 + kStageWarps - 1 (staging): per chunk, waits for its
//     pages, dequantizes K and V into the buffers the MMAs of two chunks ago
//     have released, and issues the copies of the chunk after next;
//   * warp kMmaWarp, one thread (MMA): S(i) = Q K(i)^T into one of two
//     tensor-memory score buffers as soon as K(i) is staged, then
//     O += P(i-1) V(i-1).
// Tensor memory: O in columns 0..127, the two score buffers in 128..191 and
// 192..255.  One CTA per SM (228 KB of shared memory).
template <int KF, int VF>
__global__ void __launch_bounds__(kWsThreads, 1) cascade_prefix_ws_kernel(const CascadeParams p) {
  constexpr int D = 128;
  constexpr int NC = cascade_chunk_tokens(D);       // 64 prefix tokens per chunk
  constexpr int NPG = NC / kPage;
  constexpr int NB = D / 32;
  constexpr int KSEG = k_seg_bytes(KF, D);
  constexpr int VSEG = v_seg_bytes(VF, D);
  constexpr bool kKLo = KF == MEMRA_KV_Q8_0;
  constexpr bool kVLo = VF == MEMRA_KV_Q5_1 || VF == MEMRA_KV_Q4_0;
  constexpr float kLazy = 8.f;                      // log2 units: P stays <= 256 between rescales
  // Shared memory: Q tile | K^ buffers [2] (hi, lo) | V^T buffers [2] (hi, lo)
  // | P buffers [2] | raw page buffers [2] | page ids | barriers.
  // The output rows reuse Q and the K^ buffers once the last MMA is done.
  constexpr uint32_t QB = kTileRows * D * 2, KB = NC * D * 2, VB = D * NC * 2, PB = kTileRows * NC * 2;
  constexpr uint32_t RAWB = NPG * (KSEG + VSEG);
  constexpr uint32_t OFF_Q = 0, OFF_K = QB, OFF_V = OFF_K + 4 * KB, OFF_P = OFF_V + 4 * VB, OFF_RAW = OFF_P + 2 * PB,
                     OFF_PID = OFF_RAW + 2 * RAWB;
  constexpr uint32_t ROWB = D * 4 + 16;
  constexpr uint32_t TCOLS = cascade_tmem_cols(D);
  static_assert(OFF_PID + 4 * NPG * kCascadeMaxChunksPerCta + 192 ==
                    cascade_smem_bytes(D, KSEG, VSEG, kCascadeMaxChunksPerCta), "shared-memory plan");
  static_assert(cascade_smem_bytes(D, KSEG, VSEG, kCascadeMaxChunksPerCta) <= kSmemLimit, "shared memory");
  static_assert(kTileRows * ROWB <= OFF_V, "output rows over Q and the K^ buffers");
  static_assert(D + 2 * NC <= static_cast<int>(TCOLS), "O and two score buffers fit the tensor memory");
  static_assert(KSEG % 16 == 0 && VSEG % 16 == 0 && RAWB % 16 == 0 && OFF_RAW % 16 == 0, "alignment");
  constexpr int QIT = kTileRows * (D / 8) / 256;               // Q items per thread of warps 0-7
  constexpr int KIT = NC * (D / 8) / kStageThreads;            // K items per staging thread and chunk
  constexpr int VTASKS = VF == MEMRA_KV_NVFP4 ? NPG * 2 * (D / 16) * 8 : NPG * 2 * NB * 8 * 2;
  constexpr int VIT = VTASKS / kStageThreads;                  // V tasks per staging thread and chunk
  static_assert(QIT * 256 == kTileRows * (D / 8) && KIT * kStageThreads == NC * (D / 8) &&
                    VIT * kStageThreads == VTASKS, "whole items");

  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sb = smem_addr(smem);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t OFF_BAR = OFF_PID + 4 * NPG * p.cpc;
  // barriers, two of each: raw pages landed, K^ staged / read, V^T staged / read,
  // scores written / read, P written / read
  const uint32_t bars = sb + OFF_BAR;
  auto bar = [&](int kind, int b) { return bars + 16 * kind + 8 * b; };
  enum { kRaw = 0, kKFull, kKEmpty, kVFull, kVEmpty, kSFull, kSEmpty, kPFull, kPEmpty };
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + OFF_BAR + 16 * 9);
  int *pid_s = reinterpret_cast<int *>(smem + OFF_PID);

  const int kvh = blockIdx.y;
  const int rows = p.batch * p.q_len * p.group;
  const int r0 = blockIdx.z * kTileRows;
  const int c0 = blockIdx.x * p.cpc;
  const int nck = max(0, min(p.cpc, p.n_chunks - c0));
  const int rows_per_seq = p.q_len * p.group;

  if (warp == kMmaWarp) {
    tc::tmem_alloc(smem_addr(tmem_slot), TCOLS);
    tc::tmem_relinquish();
  }
  if (tid == 32 * kMmaWarp) {
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(kRaw, b), 1);
      mbar_init(bar(kKFull, b), kStageThreads);
      mbar_init(bar(kKEmpty, b), 1);
      mbar_init(bar(kVFull, b), kStageThreads);
      mbar_init(bar(kVEmpty, b), 1);
      mbar_init(bar(kSFull, b), 1);
      mbar_init(bar(kSEmpty, b), 128);
      mbar_init(bar(kPFull, b), 128);
      mbar_init(bar(kPEmpty, b), 1);
    }
    fence_barrier_init();
  }
  grid_dependency_wait();          // q, the pools and the tables are written
  allow_dependent_launch();

  // the Q tile's loads first: their latency overlaps the page-id reads
  uint4 qv[QIT];
  if (tid < 256) {
#pragma unroll
    for (int it = 0; it < QIT; ++it) {
      const int i = tid + it * 256;
      const int rest = i >> 3, u = rest % (D / 8);
      const int r = r0 + (rest / (D / 8)) * 8 + (i & 7);
      qv[it] = make_uint4(0, 0, 0, 0);
      if (r < rows) {
        const int b = r / rows_per_seq, rem = r % rows_per_seq;
        const size_t rowid = (static_cast<size_t>(b) * p.q_len + rem / p.group) * p.n_heads + kvh * p.group +
                             rem % p.group;
        qv[it] = *reinterpret_cast<const uint4 *>(p.q + rowid * D + 8 * u);
      }
    }
  }
  for (int i = tid; i < nck * NPG; i += kWsThreads) {
    const int tok = c0 * NC + i * kPage;
    int pid = -1;
    if (tok < p.prefix_len) {
      pid = p.page_table[tok / kPage];
      if (pid < 0 || pid >= p.num_pages) {
        flag_error(p.status, MEMRA_DEVERR_BAD_PAGE);
        pid = -1;
      }
    }
    pid_s[i] = pid;
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  const size_t kstride = static_cast<size_t>(p.n_kv_heads) * KSEG, vstride = static_cast<size_t>(p.n_kv_heads) * VSEG;
  auto issue = [&](int ci) {       // chunk ci's pages into raw buffer ci % 2
    const uint32_t buf = sb + OFF_RAW + (ci & 1) * RAWB, br = bar(kRaw, ci & 1);
    uint32_t bytes = 0;
    for (int i = 0; i < NPG; ++i) bytes += pid_s[ci * NPG + i] >= 0 ? KSEG + VSEG : 0;
    if (!bytes) {
      mbar_arrive(br);
      return;
    }
    mbar_arrive_expect_tx(br, bytes);
    for (int i = 0; i < NPG; ++i) {
      const int pg = pid_s[ci * NPG + i];
      if (pg < 0) continue;
      bulk_copy_g2s_nohint(buf + i * KSEG, p.k_pool + pg * kstride + static_cast<size_t>(kvh) * KSEG, KSEG, br);
      bulk_copy_g2s_nohint(buf + NPG * KSEG + i * VSEG, p.v_pool + pg * vstride + static_cast<size_t>(kvh) * VSEG,
                           VSEG, br);
    }
  };
  auto chunk_mask = [&](int ci) {
    uint32_t m = 0;
#pragma unroll
    for (int i = 0; i < NPG; ++i) m |= (pid_s[ci * NPG + i] >= 0 ? 1u : 0u) << i;
    return m;
  };
  if (tid == 128) {
    if (nck > 0) issue(0);
    if (nck > 1) issue(1);
  }
  if (tid < 256) {
#pragma unroll
    for (int it = 0; it < QIT; ++it) sts128(sb + OFF_Q + 16 * (tid + it * 256), qv[it]);
    fence_proxy_async();           // the Q tile is read by the tensor cores
  }
  __syncthreads();

  bool ok = true;
  if (warp >= 4 && warp < kMmaWarp) {
    // ------------------------------------------------------------ staging --
    const int st = tid - 128;
    int issued = min(nck, 2), consumed = 0;
    for (int ci = 0; ci < nck && ok; ++ci) {
      const int b = ci & 1, u = ci >> 1;
      const uint32_t rawk = sb + OFF_RAW + b * RAWB, rawv = rawk + NPG * KSEG;
      const uint32_t kbuf = sb + OFF_K + b * 2 * KB, vbuf = sb + OFF_V + b * 2 * VB;
      const uint32_t pmask = chunk_mask(ci);
      ok = mbar_wait_bounded(bar(kRaw, b), u & 1, p.status);
      if (ok && ci >= 2) ok = mbar_wait_bounded(bar(kKEmpty, b), (u - 1) & 1, p.status);
      ok = staging_all(ok);        // uniform over the staging warps: every one takes the same branch
      if (!ok) break;
      consumed = ci + 1;
      {   // K^: item i = (token group, 8-dim group, token in group) at byte 16 i
        KRaw kr[KIT];
#pragma unroll
        for (int it = 0; it < KIT; ++it) {
          const int i = st + it * kStageThreads;
          const int n = ((i >> 3) / (D / 8)) * 8 + (i & 7);
          kr[it] = load_k8<D, KF>(rawk + (n / kPage) * KSEG, n % kPage, (i >> 3) % (D / 8));
        }
#pragma unroll
        for (int it = 0; it < KIT; ++it) {
          const int i = st + it * kStageThreads;
          const int n = ((i >> 3) / (D / 8)) * 8 + (i & 7);
          uint32_t hi[4] = {0, 0, 0, 0}, lo[4] = {0, 0, 0, 0};
          if ((pmask >> (n / kPage)) & 1u) convert_k8<KF>(kr[it], n % kPage, hi, lo);
          sts128(kbuf + 16 * i, make_uint4(hi[0], hi[1], hi[2], hi[3]));
          if constexpr (kKLo) sts128(kbuf + KB + 16 * i, make_uint4(lo[0], lo[1], lo[2], lo[3]));
        }
      }
      fence_proxy_async();
      mbar_arrive(bar(kKFull, b));
      if (ci >= 2) ok = mbar_wait_bounded(bar(kVEmpty, b), (u - 1) & 1, p.status);
      ok = staging_all(ok);
      if (!ok) break;
      auto vt_store = [&](int dd, int g, uint4 h, uint4 l) {
        const uint32_t off = ((dd >> 3) * (NC / 8) + g) * 128 + (dd & 7) * 16;
        sts128(vbuf + off, h);
        if constexpr (kVLo) sts128(vbuf + VB + off, l);
      };
      if constexpr (VF == MEMRA_KV_NVFP4) {
        // task (page, half page, 16-dim block b16, rr): dims 16 b16 + rr and + 8
        uint32_t cw[VIT][4], sw[VIT][4];
#pragma unroll
        for (int it = 0; it < VIT; ++it) {
          const int task = st + it * kStageThreads;
          const int rr = task & 7, b16 = (task >> 3) % (D / 16), ps = task / (16 * (D / 16));
          const uint32_t seg = rawv + ps * VSEG;
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            cw[it][c] = lds32(seg + ((b16 >> 2) * 32 + 4 * rr + c) * 16 + (b16 & 3) * 4);
            sw[it][c] = lds32(seg + 8 * D + (c * (D / 16) + b16) * 4);
          }
        }
#pragma unroll
        for (int it = 0; it < VIT; ++it) {
          const int task = st + it * kStageThreads;
          const int rr = task & 7, b16 = (task >> 3) % (D / 16), ph = (task / (8 * (D / 16))) & 1,
                    ps = task / (16 * (D / 16));
          uint32_t h0[4] = {0, 0, 0, 0}, h1[4] = {0, 0, 0, 0};
          if ((pmask >> ps) & 1u) {
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              __half2 v[2];
#pragma unroll
              for (int f = 0; f < 2; ++f) {
                const int sh = 8 * (f + 2 * ph);
                v[f] = __hmul2(bits_h2(e2m1x2_to_half2((cw[it][c] >> sh) & 0xFFu)), e4m3_scale_h2(sw[it][c] >> sh));
              }
              h0[c] = h2_bits(__lows2half2(v[0], v[1]));
              h1[c] = h2_bits(__highs2half2(v[0], v[1]));
            }
          }
          const uint4 z = make_uint4(0, 0, 0, 0);
          vt_store(16 * b16 + rr, 2 * ps + ph, make_uint4(h0[0], h0[1], h0[2], h0[3]), z);
          vt_store(16 * b16 + rr + 8, 2 * ps + ph, make_uint4(h1[0], h1[1], h1[2], h1[3]), z);
        }
      } else {
        // task (page, half page, block b, vg, pair h): dims 32 b + 4 vg + 2 h + s, tokens 8 half + 2 c + f
        VRaw vr[VIT];
#pragma unroll
        for (int it = 0; it < VIT; ++it) {
          const int task = st + it * kStageThreads;
          const int h = task & 1, vg = (task >> 1) & 7, bb = (task >> 4) % NB, ph = (task / (16 * NB)) & 1,
                    ps = task / (32 * NB);
          vr[it] = load_v_task<D, VF>(rawv + ps * VSEG, ph, bb, vg, h);
        }
#pragma unroll
        for (int it = 0; it < VIT; ++it) {
          const int task = st + it * kStageThreads;
          const int h = task & 1, vg = (task >> 1) & 7, bb = (task >> 4) % NB, ph = (task / (16 * NB)) & 1,
                    ps = task / (32 * NB);
          uint32_t hi[2][4], lo[2][4];
          convert_v_task<VF>(vr[it], ph, bb, h, hi, lo);
          const bool have = (pmask >> ps) & 1u;
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const uint4 hv = have ? make_uint4(hi[e][0], hi[e][1], hi[e][2], hi[e][3]) : make_uint4(0, 0, 0, 0);
            const uint4 lv = have && kVLo ? make_uint4(lo[e][0], lo[e][1], lo[e][2], lo[e][3]) : make_uint4(0, 0, 0, 0);
            vt_store(32 * bb + 4 * vg + 2 * h + e, 2 * ps + ph, hv, lv);
          }
        }
      }
      fence_proxy_async();         // V^T for the tensor cores; the raw buffer for the next copies
      mbar_arrive(bar(kVFull, b));
      staging_all(true);           // every staging thread is done with the raw buffer
      if (st == 0 && ci + 2 < nck) issue(ci + 2);
      issued = min(nck, ci + 3);
    }
    // after a wait that gave up, the copies still in flight land (bounded) before the CTA leaves
    if (!ok)
      for (int ci = consumed; ci < issued; ++ci) mbar_wait_bounded(bar(kRaw, ci & 1), (ci >> 1) & 1, p.status);
    // Every sequence of the row tile must hold the same prefix pages and see
    // all of the prefix.  Checked here, while the last chunk's MMAs and softmax
    // are still running (flags only; one KV head checks).
    if (kvh == 0) {
      const int b_first = r0 / rows_per_seq, b_last = (min(rows, r0 + kTileRows) - 1) / rows_per_seq;
      const int pages = nck * NPG;
      for (int i = st; i < (b_last - b_first + 1) * pages; i += kStageThreads) {
        const int bb = b_first + i / pages, j = c0 * NPG + i % pages;
        if (j * kPage < p.prefix_len && p.page_table[static_cast<size_t>(bb) * p.max_pages + j] != p.page_table[j])
          flag_error(p.status, MEMRA_DEVERR_PREFIX);
      }
      if (blockIdx.x == 0)
        for (int bb = b_first + st; bb <= b_last; bb += kStageThreads)
          if (p.seq_lens[bb] - p.q_len < p.prefix_len) flag_error(p.status, MEMRA_DEVERR_BAD_SEQ_LEN);
    }
  } else if (warp == kMmaWarp) {
    // ---------------------------------------------------------------- MMA --
    if (lane == 0) {
      constexpr uint32_t idesc_s = tc::idesc_f16_f32(kTileRows, NC);
      constexpr uint32_t idesc_o = tc::idesc_f16_f32(kTileRows, D);
      // S(i) = Q K(i)^T into score buffer i % 2, as soon as K(i) is staged and
      // the softmax has read S(i - 2) there
      auto mma_s = [&](int i) {
        const int bb = i & 1, u = i >> 1;
        ok = mbar_wait_bounded(bar(kKFull, bb), u & 1, p.status);
        if (ok && i >= 2) ok = mbar_wait_bounded(bar(kSEmpty, bb), (u - 1) & 1, p.status);
        if (!ok) return;
        tc::fence_after_sync();
        const uint32_t kbuf = sb + OFF_K + bb * 2 * KB;
#pragma unroll 1
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint64_t a = tc::smem_desc(sb + OFF_Q + 256 * ks, 128, (D / 8) * 128);
          tc::mma_f16(tmem + D + bb * NC, a, tc::smem_desc(kbuf + 256 * ks, 128, (D / 8) * 128), idesc_s, ks > 0);
          if constexpr (kKLo)
            tc::mma_f16(tmem + D + bb * NC, a, tc::smem_desc(kbuf + KB + 256 * ks, 128, (D / 8) * 128), idesc_s, 1);
        }
        tc::commit(bar(kKEmpty, bb));
        tc::commit(bar(kSFull, bb));
      };
      // O += P(j) V(j) once the softmax has written P(j) and V(j) is staged
      auto mma_o = [&](int j) {
        const int bb = j & 1, u = j >> 1;
        ok = mbar_wait_bounded(bar(kPFull, bb), u & 1, p.status);
        if (ok) ok = mbar_wait_bounded(bar(kVFull, bb), u & 1, p.status);
        if (!ok) return;
        tc::fence_after_sync();
        const uint32_t pbuf = sb + OFF_P + bb * PB, vbuf = sb + OFF_V + bb * 2 * VB;
#pragma unroll 1
        for (int ks = 0; ks < NC / 16; ++ks) {
          const uint64_t a = tc::smem_desc(pbuf + 256 * ks, 128, (NC / 8) * 128);
          tc::mma_f16(tmem, a, tc::smem_desc(vbuf + 256 * ks, 128, (NC / 8) * 128), idesc_o, j > 0 || ks > 0);
          if constexpr (kVLo)
            tc::mma_f16(tmem, a, tc::smem_desc(vbuf + VB + 256 * ks, 128, (NC / 8) * 128), idesc_o, 1);
        }
        tc::commit(bar(kVEmpty, bb));
        tc::commit(bar(kPEmpty, bb));
      };
      // the scores run two chunks ahead of the output, so that the softmax of
      // chunk j + 1 finds its scores ready while P(j) V(j) is computed
      if (nck > 0) mma_s(0);
      if (ok && nck > 1) mma_s(1);
      for (int j = 0; j < nck && ok; ++j) {
        mma_o(j);
        if (ok && j + 2 < nck) mma_s(j + 2);
      }
    }
  } else {
    // ------------------------------------------------------------ softmax --
    const int rl = tid;                                   // row of the tile, tensor-memory lane
    const uint32_t tlane = static_cast<uint32_t>(warp * 32) << 16;
    float m_row = -INFINITY, l_row = 0.f;
    for (int ci = 0; ci < nck && ok; ++ci) {
      const int b = ci & 1, u = ci >> 1;
      const uint32_t pmask = chunk_mask(ci);
      ok = mbar_wait_bounded(bar(kSFull, b), u & 1, p.status);
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      tc::fence_after_sync();
      uint32_t sr[NC];
#pragma unroll
      for (int k0 = 0; k0 < NC; k0 += 16) tc::ld_32x32b_x16(tmem + tlane + D + b * NC + k0, sr + k0);
#pragma unroll
      for (int k0 = 0; k0 < NC; k0 += 16) tc::wait_ld(sr + k0);
      tc::fence_before_sync();
      mbar_arrive(bar(kSEmpty, b));
      float m_chunk = -INFINITY;
#pragma unroll
      for (int k = 0; k < NC; ++k) {
        const bool valid = (pmask >> (k / kPage)) & 1u;
        const float v = valid ? __uint_as_float(sr[k]) * p.scale_log2 : -INFINITY;
        sr[k] = __float_as_uint(v);
        m_chunk = fmaxf(m_chunk, v);
      }
      float alpha = 1.f;
      if (m_chunk > m_row + kLazy) {         // also the first chunk with a key (m_row = -inf)
        if (m_row != -INFINITY) alpha = fast_exp2(m_row - m_chunk);
        m_row = m_chunk;
      }
      if (ci > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
        // O must be quiescent: the output MMA of the previous chunk is done
        ok = mbar_wait_bounded(bar(kPEmpty, (ci - 1) & 1), ((ci - 1) >> 1) & 1, p.status);
        if (!__all_sync(0xffffffffu, ok)) {
          ok = false;
          break;
        }
        tc::fence_after_sync();
#pragma unroll 1
        for (int k0 = 0; k0 < D; k0 += 16) {
          uint32_t orr[16];
          tc::ld_32x32b_x16(tmem + tlane + k0, orr);
          tc::wait_ld(orr);
#pragma unroll
          for (int e = 0; e < 16; ++e) orr[e] = __float_as_uint(__uint_as_float(orr[e]) * alpha);
          tc::st_32x32b_x16(tmem + tlane + k0, orr);
        }
        tc::wait_st();
      }
      // P buffer ci % 2 is free once the output MMA of chunk ci - 2 is done
      if (ci >= 2) ok = mbar_wait_bounded(bar(kPEmpty, b), (u - 1) & 1, p.status);
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      const uint32_t pbuf = sb + OFF_P + b * PB;
      float lsum = 0.f;
#pragma unroll
      for (int g = 0; g < NC / 8; ++g) {
        uint32_t w4[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float p0 = m_row == -INFINITY ? 0.f : fast_exp2(__uint_as_float(sr[8 * g + 2 * e]) - m_row);
          const float p1 = m_row == -INFINITY ? 0.f : fast_exp2(__uint_as_float(sr[8 * g + 2 * e + 1]) - m_row);
          const __half2 ph2 = __floats2half2_rn(p0, p1);
          const float2 back = __half22float2(ph2);
          lsum += back.x + back.y;
          w4[e] = h2_bits(ph2);
        }
        sts128(pbuf + ((rl >> 3) * (NC / 8) + g) * 128 + (rl & 7) * 16, make_uint4(w4[0], w4[1], w4[2], w4[3]));
      }
      l_row = l_row * alpha + lsum;
      fence_proxy_async();
      tc::fence_before_sync();
      mbar_arrive(bar(kPFull, b));
    }
    // the last output MMA done: o = O * v_post / l into padded rows (Q and the K^ buffers are free)
    if (ok && nck > 0) ok = mbar_wait_bounded(bar(kPEmpty, (nck - 1) & 1), ((nck - 1) >> 1) & 1, p.status);
    bool wrote = false;
    if (__all_sync(0xffffffffu, ok) && nck > 0) {
      tc::fence_after_sync();
      const float inv = l_row > 0.f ? p.v_post / l_row : 0.f;
#pragma unroll 1
      for (int k0 = 0; k0 < D; k0 += 32) {
        uint32_t orr[32];
        tc::ld_32x32b_x16(tmem + tlane + k0, orr);
        tc::ld_32x32b_x16(tmem + tlane + k0 + 16, orr + 16);
        tc::wait_ld(orr);
        tc::wait_ld(orr + 16);
#pragma unroll
        for (int e = 0; e < 32; e += 4)
          sts128(sb + OFF_Q + rl * ROWB + (k0 + e) * 4,
                 l_row > 0.f ? make_uint4(__float_as_uint(__uint_as_float(orr[e]) * inv),
                                          __float_as_uint(__uint_as_float(orr[e + 1]) * inv),
                                          __float_as_uint(__uint_as_float(orr[e + 2]) * inv),
                                          __float_as_uint(__uint_as_float(orr[e + 3]) * inv))
                             : make_uint4(0, 0, 0, 0));
      }
      wrote = true;
    }
    // This CTA's partial of the row: the row by one bulk copy of the padded
    // shared-memory row this thread wrote, the lse by a plain store.  A row
    // without keys, or every row after a wait that gave up, gets lse = -inf,
    // which the merge never weighs.
    if (r0 + rl < rows) {
      const size_t slot = prefix_row_id(p, kvh, r0 + rl) * p.n_parts + blockIdx.x;
      if (wrote) {
        fence_proxy_async();
        bulk_store_s2g(p.o_pre + slot * D, sb + OFF_Q + rl * ROWB, D * 4);
      }
      p.lse_pre[slot] = wrote && l_row > 0.f ? m_row + __log2f(l_row) : -INFINITY;
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == kMmaWarp) tc::tmem_dealloc(tmem, TCOLS);
  bulk_store_wait();               // the row copies this thread issued (none: returns at once)
}

// Merge of a row's prefix-chunk partials and its own-key split partials.
template <int D>
__global__ void __launch_bounds__(kThreads) cascade_combine_kernel(const CascadeCombineParams p) {
  constexpr int PER = D / 32;
  constexpr int W = kThreads / 32;
  __shared__ float red[W][D];
  __shared__ float redl[W];
  __shared__ float mx[W];
  const int row = blockIdx.x, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b = row / (p.q_len * p.n_heads), qi = (row / p.n_heads) % p.q_len;
  // the row's own-key plan before the wait: the lengths were complete before
  // the call's first pass started
  const int Tseq = clamp_seq_len(p.seq_lens[b], p.q_len, p.max_seq_len, p.max_pages, false, p.status, false);
  const int ns = min(key_range(Tseq, p.q_len, qi, 0, p.prefix_len, p.split_target).ns, p.nsplit_max);
  grid_dependency_wait();          // both passes are complete
  const int parts = p.n_parts + ns;
  auto lse_of = [&](int k) {
    return k < p.n_parts ? p.lse_pre[static_cast<size_t>(row) * p.n_parts + k]
                         : p.lse_suf[static_cast<size_t>(row) * p.nsplit_max + (k - p.n_parts)];
  };
  auto o_of = [&](int k) {
    return k < p.n_parts ? p.o_pre + (static_cast<size_t>(row) * p.n_parts + k) * D
                         : p.o_suf + (static_cast<size_t>(row) * p.nsplit_max + (k - p.n_parts)) * D;
  };
  // One pass: warp w takes parts w, w + W, ..., eight in flight at a time,
  // their lse and rows loaded together, and keeps a running maximum (its
  // partial sums rescaled when it moves).  A part with lse = -inf (no keys, or
  // a CTA that gave up) is never weighed: its row may hold anything.
  float mw = -INFINITY, L = 0.f;
  float acc[PER];
#pragma unroll
  for (int e = 0; e < PER; ++e) acc[e] = 0.f;
  constexpr int BATCH = 8;
  for (int k0 = warp; k0 < parts; k0 += BATCH * W) {
    float ls[BATCH];
    float4 x[BATCH][PER / 4];
#pragma unroll
    for (int u = 0; u < BATCH; ++u) {
      const int k = k0 + u * W;
      const bool in = k < parts;
      ls[u] = in ? lse_of(k) : -INFINITY;
      const float4 *src = reinterpret_cast<const float4 *>(o_of(in ? k : 0) + lane * PER);
#pragma unroll
      for (int q4 = 0; q4 < PER / 4; ++q4) x[u][q4] = in ? src[q4] : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int u = 0; u < BATCH; ++u) {
      if (ls[u] == -INFINITY) continue;
      if (ls[u] > mw) {
        const float sc = fast_exp2(mw - ls[u]);      // 0 while mw = -inf
        L *= sc;
#pragma unroll
        for (int e = 0; e < PER; ++e) acc[e] *= sc;
        mw = ls[u];
      }
      const float wgt = fast_exp2(ls[u] - mw);
      L += wgt;
#pragma unroll
      for (int q4 = 0; q4 < PER / 4; ++q4) {
        acc[4 * q4 + 0] = fmaf(wgt, x[u][q4].x, acc[4 * q4 + 0]);
        acc[4 * q4 + 1] = fmaf(wgt, x[u][q4].y, acc[4 * q4 + 1]);
        acc[4 * q4 + 2] = fmaf(wgt, x[u][q4].z, acc[4 * q4 + 2]);
        acc[4 * q4 + 3] = fmaf(wgt, x[u][q4].w, acc[4 * q4 + 3]);
      }
    }
  }
#pragma unroll
  for (int e = 0; e < PER; ++e) red[warp][lane * PER + e] = acc[e];
  if (lane == 0) {
    redl[warp] = L;
    mx[warp] = mw;
  }
  __syncthreads();
  // the warps' sums, each scaled from its own maximum to the row's
  float M = mx[0];
#pragma unroll
  for (int w = 1; w < W; ++w) M = fmaxf(M, mx[w]);
  float wscale[W];
#pragma unroll
  for (int w = 0; w < W; ++w) wscale[w] = mx[w] == -INFINITY ? 0.f : fast_exp2(mx[w] - M);
  __half *dst = p.out + static_cast<size_t>(row) * D;
  for (int j = threadIdx.x; j < D / 2; j += kThreads) {
    float a0 = 0.f, a1 = 0.f, l = 0.f;
#pragma unroll
    for (int w = 0; w < W; ++w) {
      a0 = fmaf(wscale[w], red[w][2 * j], a0);
      a1 = fmaf(wscale[w], red[w][2 * j + 1], a1);
      l = fmaf(wscale[w], redl[w], l);
    }
    const float inv = l > 0.f ? 1.f / l : 0.f;
    reinterpret_cast<__half2 *>(dst)[j] = __floats2half2_rn(a0 * inv, a1 * inv);
  }
}

// The prefix-pass kernel of a head_dim: warp-specialized at 128, generic at 256.
template <int D, int KF, int VF>
constexpr auto prefix_kernel() {
  if constexpr (D == 128)
    return cascade_prefix_ws_kernel<KF, VF>;
  else
    return cascade_prefix_kernel<D, KF, VF>;
}

template <int D, int KF, int VF>
cudaError_t wave_one(int *wave_ctas) {
  constexpr uint32_t smem_max = cascade_smem_bytes(D, k_seg_bytes(KF, D), v_seg_bytes(VF, D), kCascadeMaxChunksPerCta);
  // any mix of prefix-pass CTAs that fits an SM by shared memory fits its tensor memory
  constexpr uint32_t kMin128 = cascade_smem_bytes(128, 9 * 128, 9 * 128, 1) + 1024u;   // smallest CTAs
  constexpr uint32_t kMin256 = cascade_smem_bytes(256, 9 * 256, 9 * 256, 1) + 1024u;
  static_assert(2u * kMin128 > 233472u && 2u * kMin256 > 233472u && kMin256 + kMin128 > 233472u &&
                    cascade_tmem_cols(128) <= 512u && cascade_tmem_cols(256) <= 512u,
                "one prefix-pass CTA per SM, whatever the head_dim");
  auto kernel = prefix_kernel<D, KF, VF>();
  // Per device and instantiation: the CTAs one wave holds, the SMs times the
  // CTAs per SM the kernel is built for (one).  It depends on the device only,
  // never on the batch.  The kernel's shared-memory limit is set here once.
  static int wave[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!wave[dev]) {
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem_max));
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    int sms = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    wave[dev] = std::max(1, sms * cascade_ctas_per_sm(D));
  }
  *wave_ctas = wave[dev];
  return cudaSuccess;
}

template <int D, int KF, int VF>
cudaError_t launch_prefix_one(CascadeParams &p, cudaStream_t st) {
  int wave = 1;
  cudaError_t e = wave_one<D, KF, VF>(&wave);     // also sets the shared-memory limit once
  if (e != cudaSuccess) return e;
  const uint32_t smem = cascade_smem_bytes(D, k_seg_bytes(KF, D), v_seg_bytes(VF, D), p.cpc);
  auto kernel = prefix_kernel<D, KF, VF>();
  p.n_parts = (p.n_chunks + p.cpc - 1) / p.cpc;      // CTAs per (KV head, row tile): one partial each
  const int rows = p.batch * p.q_len * p.group;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(p.n_parts), static_cast<unsigned>(p.n_kv_heads),
                     static_cast<unsigned>((rows + kTileRows - 1) / kTileRows));
  cfg.blockDim = dim3(D == 128 ? kWsThreads : kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const CascadeParams args = p;
  return cudaLaunchKernelEx(&cfg, kernel, args);
}

template <int D>
cudaError_t wave_formats(int kf, int vf, int *wave_ctas) {
  auto by_v = [&](auto kc) -> cudaError_t {
    constexpr int K = decltype(kc)::value;
    switch (vf) {
      case MEMRA_KV_Q5_1: return wave_one<D, K, MEMRA_KV_Q5_1>(wave_ctas);
      case MEMRA_KV_Q4_0: return wave_one<D, K, MEMRA_KV_Q4_0>(wave_ctas);
      case MEMRA_KV_FP8_E4M3: return wave_one<D, K, MEMRA_KV_FP8_E4M3>(wave_ctas);
      case MEMRA_KV_NVFP4: return wave_one<D, K, MEMRA_KV_NVFP4>(wave_ctas);
      default: return cudaErrorInvalidValue;
    }
  };
  switch (kf) {
    case MEMRA_KV_Q8_0: return by_v(std::integral_constant<int, MEMRA_KV_Q8_0>{});
    case MEMRA_KV_FP8_E4M3: return by_v(std::integral_constant<int, MEMRA_KV_FP8_E4M3>{});
    case MEMRA_KV_NVFP4: return by_v(std::integral_constant<int, MEMRA_KV_NVFP4>{});
    default: return cudaErrorInvalidValue;
  }
}

template <int D>
cudaError_t prefix_formats(int kf, int vf, CascadeParams &p, cudaStream_t st) {
  auto by_v = [&](auto kc) -> cudaError_t {
    constexpr int K = decltype(kc)::value;
    switch (vf) {
      case MEMRA_KV_Q5_1: return launch_prefix_one<D, K, MEMRA_KV_Q5_1>(p, st);
      case MEMRA_KV_Q4_0: return launch_prefix_one<D, K, MEMRA_KV_Q4_0>(p, st);
      case MEMRA_KV_FP8_E4M3: return launch_prefix_one<D, K, MEMRA_KV_FP8_E4M3>(p, st);
      case MEMRA_KV_NVFP4: return launch_prefix_one<D, K, MEMRA_KV_NVFP4>(p, st);
      default: return cudaErrorInvalidValue;
    }
  };
  switch (kf) {
    case MEMRA_KV_Q8_0: return by_v(std::integral_constant<int, MEMRA_KV_Q8_0>{});
    case MEMRA_KV_FP8_E4M3: return by_v(std::integral_constant<int, MEMRA_KV_FP8_E4M3>{});
    case MEMRA_KV_NVFP4: return by_v(std::integral_constant<int, MEMRA_KV_NVFP4>{});
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_cascade_prefix(int D, int kf, int vf, CascadeParams &p, cudaStream_t st) {
  if (p.n_chunks == 0 || p.batch == 0) return cudaSuccess;
  return D == 128 ? prefix_formats<128>(kf, vf, p, st) : prefix_formats<256>(kf, vf, p, st);
}

cudaError_t cascade_wave(int D, int kf, int vf, int *wave_ctas) {
  return D == 128 ? wave_formats<128>(kf, vf, wave_ctas) : wave_formats<256>(kf, vf, wave_ctas);
}

cudaError_t launch_cascade_combine(int D, const CascadeCombineParams &p, cudaStream_t st) {
  if (p.rows == 0) return cudaSuccess;
  const dim3 grid(static_cast<unsigned>(p.rows)), block(kThreads);
  if (D == 128) return launch_pdl(cascade_combine_kernel<128>, grid, block, 0, st, p);
  return launch_pdl(cascade_combine_kernel<256>, grid, block, 0, st, p);
}

}  // namespace memra
