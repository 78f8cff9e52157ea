// K2: split-K flash-decoding over the block-quantized paged KV cache.
//
// What it computes: for one (sequence, KV head, query position, group of up
// to 8 query heads, split of C(T) tokens), the partial softmax(q K^T * scale) V
// over the split's keys, as (o = O / l, lse = m + log2 l); T is the number of
// keys the position sees (causal among the q_len new tokens).  The KV formats
// are the memra-bench card's knobs (section "drafts/kf4/ - archived
// experiment"); plain decode and MTP verify are the memra README's
// "Speculative decoding" item; the 262,144-token contexts its "Long context
// and larger models" item.
//
// Every query position is planned as its own decode problem: its split size
// C(T) comes from its own T, its CTAs see exactly the keys a q_len = 1 call at
// that position sees, and nothing in a row's arithmetic depends on the other
// rows of the call.  So verify rows are byte-identical to plain decode at the
// same positions (the README's single numeric class for speculative decode).
// The CTAs of one split's positions are neighbours in the grid and read the
// same pages, so L2 serves all but the first read.
//
// How (one CTA = 8 warps at head_dim 128, 2 CTAs per SM; 4 warps at 256, 3 per SM):
//  * Warp w takes pages w, w + W, ... of the split, issues its own pages'
//    copies (one contiguous bulk copy each for the K and V segments, 16-byte
//    aligned, evict-first in L2) `num_stages` pages ahead into its own ring
//    stages, completing on per-stage mbarriers, and refills a stage once read.
//    Per page: S^T[16 tokens x 8 rows] = K^ Q^T on the tensor cores
//    (m16n8k16, fp16 in, fp32 out) with the K codes converted to fp16 in
//    registers; the q8_0 block scale multiplies each 32-element block's
//    partial sum, so K^ is exact.  Online softmax in the fp32 accumulators
//    (row max over the 8 token lanes by xor-shuffles), P transposed in
//    registers (movmatrix) into the B operand, then O^T[D x rows] += V^T P^T
//    with the V codes converted in registers and the per-token block scale
//    folded into P; q5_1's +m term is one extra MMA (blocks x tokens) * P^T.
//  * q8_0 K codes are stored biased (q + 128) and become fp16 1152 + q with
//    one byte permute per pair; one more MMA per page, with the block scales
//    as A and -1152 * sum(Q) as B (fp16 hi + lo), takes the bias out.
//  * The reference maximum of a row moves only when a score passes it by more
//    than 2 (log2 units), so O and l are rescaled only then.
//  * At the end the warps merge their (m, l, O) through shared memory; a
//    split that covers all of the position's keys writes fp16 output,
//    otherwise an fp32 partial for the combine kernel.
//  * Fused append (memra_decode_step): the step's new K/V rows that the CTA
//    sees are quantized and stored into their pages before those pages are
//    copied in.
// Every wait is bounded (MEMRA_DEVERR_TIMEOUT); bad page ids are skipped
// (MEMRA_DEVERR_BAD_PAGE); keys past T never reach the result, even if their
// bytes are garbage.
#pragma once

#include <cuda_runtime.h>

#include <type_traits>

#include "kv_quant.cuh"

namespace memra {

struct DecodeParams {
  const uint8_t *k_pool;
  const uint8_t *v_pool;
  const __half *q;
  const int32_t *page_table;
  const int32_t *seq_lens;
  __half *out;
  float *o_part;      // [rows][nsplit_max][D]
  float *lse_part;    // [rows][nsplit_max]
  int32_t *status;
  // Fused append (null when the step's rows are already in the pools): the
  // K and V rows of the q_len new tokens, fp16 [batch][q_len][n_kv_heads][D],
  // stored at positions seq_len - q_len .. seq_len - 1 before they are read.
  const __half *k_new;
  const __half *v_new;
  int n_kv_heads, num_pages, max_pages, max_seq_len, q_len, n_heads, group;
  int window;         // sliding window in tokens, 0 = none
  int skip;           // keys below this are another pass's (a shared prefix): not read, and every
                      // split writes its partial so that the passes can be merged
  int ring;           // 1: page_table rows are rings of max_pages columns (position p -> (p / 16) % max_pages)
  int ngh;            // groups of 8 query heads per KV head: ceil(group / 8)
  int ngh_q;          // CTAs per (split, KV head, sequence): q_len * ngh
  int nsplit_max, num_stages, split_target;
  float scale_log2, v_scale, k_scale;
  // Test hooks of the bounded waits (memra_testing.h); kWaitLimitNs and 0 in
  // every other call.  page_wait_ns bounds the waits for pages in the main
  // loop; test_extra_tx > 0 makes CTA (0, 0, 0) expect that many bytes more
  // than the copies of its first page deliver, so that page's wait runs out.
  unsigned long long page_wait_ns;
  int test_extra_tx;
};

struct CombineParams {
  const int32_t *seq_lens;
  const float *o_part;
  const float *lse_part;
  __half *out;
  int32_t *status;
  int rows, q_len, n_heads, max_seq_len, max_pages, nsplit_max, split_target;
  int window, ring;
};

cudaError_t launch_combine(int D, const CombineParams &p, cudaStream_t st);
cudaError_t launch_kv_append(const memra_kv_cache &c, const void *k, const void *v, const int32_t *slots, int n_tok,
                             cudaStream_t stream);

// Warps (page lanes) per CTA: 8 at head_dim 128, 4 at 256.
template <int D>
constexpr int kWarpsFor = D == 128 ? 8 : 4;
// CTAs per SM the plan sizes shared memory and registers for: two 8-warp CTAs
// at head_dim 128; three 4-warp CTAs at 256, whose warps share one copy of
// the query fragments (12 warps per SM instead of 8 with two CTAs: the format
// sweep's split kernel 170-184 against 188-205 us, same box).
template <int D>
constexpr int kCtasPerSmFor = D == 128 ? 2 : 3;
template <int D>
constexpr bool kSharedQFor = D == 256;

template <int D>
struct MergeLayout {
  static constexpr int kW = kWarpsFor<D>;
  static constexpr int kRowsW = 8;
  static constexpr int kNb = D / 32;
  static constexpr int kO = kW * kRowsW * D;          // floats
  static constexpr int kM = kW * kRowsW;
  static constexpr int kTerm = kW * kRowsW * kNb;
  static constexpr int kBytes = (kO + 2 * kM + kTerm) * 4;
};

// Context length after the same clamping the combine kernel applies.  A
// linear page table bounds it by its columns; a ring does not.
__device__ __forceinline__ int clamp_seq_len(int T, int q_len, int max_seq_len, int max_pages, bool ring,
                                             int32_t *status, bool report) {
  int Tc = min(T, max_seq_len);
  if (!ring) Tc = min(Tc, max_pages * kPage);
  Tc = max(Tc, 0);
  if (report && (Tc != T || T < q_len)) flag_error(status, MEMRA_DEVERR_BAD_SEQ_LEN);
  return Tc;
}

// The keys a query position sees and how they are split; the split kernel and
// the combine derive it from the same numbers.
struct KeyRange {
  int T;      // one past the last visible key (the position + 1)
  int lo;     // first visible key: the window's start or the skipped prefix, else 0
  int base;   // lo rounded down to its page: splits start here
  int C;      // split size
  int ns;     // splits
};

__device__ __forceinline__ KeyRange key_range(int Tseq, int q_len, int qi, int window, int skip,
                                              int split_target) {
  KeyRange k;
  k.T = Tseq - q_len + qi + 1;
  k.lo = max(window > 0 ? k.T - window : 0, skip);
  k.lo = max(k.lo, 0);
  k.base = k.lo & ~(kPage - 1);
  const int L = k.T - k.base;
  k.C = split_tokens(L, split_target, skip > 0 ? kCascadeSplitTokens : kSplitTokens);
  k.ns = k.T > 0 && L > 0 ? (L + k.C - 1) / k.C : 0;
  return k;
}

template <int KF>
__device__ __forceinline__ void k_pairs(uint32_t w, uint32_t &lo, uint32_t &hi) {
  if constexpr (KF == MEMRA_KV_Q8_0) {
    // stored codes are q + 128: splice under the exponent of 1024 -> 1152 + q
    lo = __byte_perm(w, 0x64646464u, 0x4140);
    hi = __byte_perm(w, 0x64646464u, 0x4342);
  } else {
    e4m3x4_to_half2x2(w, lo, hi);
  }
}

template <int SH>
__device__ __forceinline__ uint32_t shift_const(uint32_t x) {
  if constexpr (SH >= 0) return x >> SH;
  else return x << (-SH);
}

template <int D, int KF, int VF>
__global__ void __launch_bounds__(kWarpsFor<D> * 32, kCtasPerSmFor<D>)
    decode_split_kernel(const DecodeParams p) {
  constexpr int NT = 1;                       // one n-tile of 8 query rows
  constexpr int NB = D / 32;
  constexpr int KSEG = k_seg_bytes(KF, D);
  constexpr int VSEG = v_seg_bytes(VF, D);
  constexpr int STAGE = KSEG + VSEG;
  using ML = MergeLayout<D>;
  constexpr int kWarps = kWarpsFor<D>;
  constexpr int kThreads = kWarps * 32;
  constexpr int ROWS_W = ML::kRowsW;
  constexpr bool kQ5 = VF == MEMRA_KV_Q5_1;
  constexpr bool kQ4 = VF == MEMRA_KV_Q4_0;
  constexpr bool kVq = kQ5 || kQ4;
  constexpr bool kK8 = KF == MEMRA_KV_Q8_0;
  constexpr bool kK4 = KF == MEMRA_KV_NVFP4;
  constexpr bool kV4 = VF == MEMRA_KV_NVFP4;
  constexpr float kLazy = 2.f;

  extern __shared__ __align__(128) uint8_t smem[];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int NS = p.num_stages;                  // a multiple of the warp count: page i and i + NS share a warp
  const int region = max(NS * STAGE, ML::kBytes);
  const uint32_t ring = smem_addr(smem);
  const uint32_t full0 = ring + region;
  int *pid_s = reinterpret_cast<int *>(smem + region + 16 * NS);   // page ids of this split, -1 = bad
  if (tid == 0) {
    for (int s = 0; s < NS; ++s) mbar_init(full0 + 8 * s, 1);
    fence_barrier_init();
  }
  // Inputs written by the launch before this one have landed.  A cascade
  // call's own-key pass (skip > 0) runs beside the prefix pass launched just
  // before it instead: it reads nothing that pass writes, and the call's
  // inputs were complete before that pass let it start.  One of its CTAs waits
  // for that pass before leaving, so this grid completes after it and the
  // merge launched after this grid sees both; the other CTAs leave as soon as
  // they are done and free their SM for the rest of the grid.
  if (p.skip == 0) grid_dependency_wait();
  // The next launch (the combine, or a cascade call's merge) may start as soon
  // as every CTA of this grid has started: its CTAs take the SMs this grid
  // frees and wait on the device for this grid to complete, so its launch
  // latency overlaps this grid's work.
  allow_dependent_launch();
  const bool waits_for_prefix = p.skip != 0 && blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0;

  // This CTA: query position qi of sequence b and query heads 8 hg .. 8 hg + 7
  // of KV head kvh's group, over the keys visible to position qi (the first
  // T of the sequence), split s of that range.  Each query position is its
  // own decode problem, planned from its own length exactly as a q_len = 1
  // call at that position would be.
  const int vr = blockIdx.x % p.ngh_q, split = blockIdx.x / p.ngh_q;
  const int qi = vr / p.ngh, hg = vr % p.ngh;
  const int kvh = blockIdx.y, b = blockIdx.z;
  const int Tseq = clamp_seq_len(p.seq_lens[b], p.q_len, p.max_seq_len, p.max_pages, p.ring, p.status,
                                 blockIdx.x == 0 && kvh == 0 && tid == 0);
  const KeyRange kr = key_range(Tseq, p.q_len, qi, p.window, p.skip, p.split_target);
  const int T = kr.T, lo = kr.lo, C = kr.C;
  if (T <= 0 || split >= kr.ns) {
    // A row with no visible key is zeros; split 0's CTA writes them, so that a
    // call whose rows all fit one split needs no combine launch.
    if (T <= 0 && split == 0 && p.skip == 0) {
      const int nr = min(8, p.group - 8 * hg);
      for (int i = tid; i < nr * (D / 8); i += kWarpsFor<D> * 32) {
        const int head = kvh * p.group + 8 * hg + i / (D / 8);
        const size_t rowid = (static_cast<size_t>(b) * p.q_len + qi) * p.n_heads + head;
        *reinterpret_cast<uint4 *>(p.out + rowid * D + 8 * (i % (D / 8))) = make_uint4(0, 0, 0, 0);
      }
    }
    if (waits_for_prefix) grid_dependency_wait();
    return;
  }
  const int tok0 = kr.base + split * C;
  const int npages = (min(T, tok0 + C) - tok0 + kPage - 1) / kPage;
  const int nsplit_b = kr.ns;
  const int nrows = min(8, p.group - 8 * hg);   // query heads of this CTA
  const int R = kWarps;                         // page lanes: warp r takes pages r, r + R, ...
  const int r = warp;

  const int g = lane >> 2, c = lane & 3;
  // The query's loads go out first: their latency overlaps the page-table reads.
  // Q^T fragments (B operand of S^T = K^ Q^T): row g, dims 32bb+8c..+7.
  uint4 qf[NT][NB];
#pragma unroll
  for (int n = 0; n < NT; ++n) {
    if (g < nrows) {
      const int head = kvh * p.group + 8 * hg + g;
      const uint4 *src = reinterpret_cast<const uint4 *>(
          p.q + ((static_cast<size_t>(b) * p.q_len + qi) * p.n_heads + head) * D + 8 * c);
#pragma unroll
      for (int bb = 0; bb < NB; ++bb) qf[n][bb] = src[4 * bb];
    } else {
#pragma unroll
      for (int bb = 0; bb < NB; ++bb) qf[n][bb] = make_uint4(0, 0, 0, 0);
    }
  }

  {
    const int32_t *pt = p.page_table + static_cast<size_t>(b) * p.max_pages;
    for (int i = tid; i < npages; i += kThreads) {
      const int j = tok0 / kPage + i;                 // logical page of the sequence
      const int pid = pt[p.ring ? j % p.max_pages : j];
      const bool ok = pid >= 0 && pid < p.num_pages;
      if (!ok) flag_error(p.status, MEMRA_DEVERR_BAD_PAGE);
      pid_s[i] = ok ? pid : -1;
    }
  }
  __syncthreads();

  // Copies of page i into stage i % NS: one bulk copy each for the K and V
  // segments, or a plain arrival for a skipped (bad) page.
  const uint64_t pol = l2_policy_evict_first();
  const uint8_t *kbase = p.k_pool + static_cast<size_t>(kvh) * KSEG;
  const uint8_t *vbase = p.v_pool + static_cast<size_t>(kvh) * VSEG;
  const size_t kstride = static_cast<size_t>(p.n_kv_heads) * KSEG;
  const size_t vstride = static_cast<size_t>(p.n_kv_heads) * VSEG;
  auto issue = [&](int i, int s) {      // page i into stage s
    const int pid = pid_s[i];
    const uint32_t bar = full0 + 8 * s;
    if (pid >= 0) {
      const bool short_page = p.test_extra_tx > 0 && i == 0 && blockIdx.x == 0 && blockIdx.y == 0 &&
                              blockIdx.z == 0;
      mbar_arrive_expect_tx(bar, STAGE + (short_page ? p.test_extra_tx : 0));
      bulk_copy_g2s(ring + s * STAGE, kbase + static_cast<size_t>(pid) * kstride, KSEG, bar, pol);
      bulk_copy_g2s(ring + s * STAGE + KSEG, vbase + static_cast<size_t>(pid) * vstride, VSEG, bar, pol);
    } else {
      mbar_arrive(bar);
    }
  };
  // New tokens of this step that this CTA sees and that fall in this split
  // (fused append only): their pages [app_lo, app_hi] are copied in only after
  // the rows are stored.  CTAs of later positions store the same rows again
  // (same bytes); each orders its own stores before its own copies.
  const int app_pos0 = max(max(Tseq - p.q_len, tok0), 0);
  const int app_n = p.k_new ? max(min(T, tok0 + C) - app_pos0, 0) : 0;
  const int app_lo = app_n ? app_pos0 / kPage - tok0 / kPage : npages;
  const int app_hi = app_n ? (app_pos0 + app_n - 1) / kPage - tok0 / kPage : -1;
  if (lane == 0) {
    for (int i = r; i < min(NS, npages); i += R)
      if (i < app_lo || i > app_hi) issue(i, i);
  }

  // Q^T fragments live in shared memory (fragment order: one conflict-free
  // 16-byte load per block), not in 16+ registers: warp-private at head_dim
  // 128, one copy per CTA (written by warp 0) at 256.
  const uint32_t qsm = smem_addr(smem + region + 16 * NS + 4 * kSplitPagesMax) + (kSharedQFor<D> ? 0 : warp * (NT * NB * 512));

  // q8_0 codes are stored biased (q + 128) and enter the MMA as fp16 1152 + q,
  // so block b's raw product is acc_b = sum_j q_j Q_j + 1152 sum_j Q_j.  The
  // bias term of a token's score, sum_b d_b * 1152 * sumQ_b, is itself a small
  // product [16 tokens x blocks] x [blocks x rows]: one more MMA per page with
  // A = the page's block scales and B = -1152 sumQ_b split into fp16 hi + lo
  // parts (k slots 0..nb-1 hi, nb..2nb-1 lo), exact to ~2^-22.
  // 1152 sumQ_b must stay inside fp16's range: a row whose block sums pass 32
  // in magnitude enters the MMAs as Q 2^-e (e >= 1, the fewest that bring them
  // to 32 or below), and its fp32 score scale takes the 2^e back.  e depends
  // on the row's own query only; ordinary queries (|sum| <= 32) keep e = 0.
  uint32_t corrb[NT][2];
  float row_scale[NT][2] = {};     // fp32 score scale of rows 8n + 2c, 8n + 2c + 1
  if constexpr (kK8) {
#pragma unroll
    for (int n = 0; n < NT; ++n) {
      auto block_sum = [&](int bb) {
        const __half2 *h = reinterpret_cast<const __half2 *>(&qf[n][bb]);
        float2 a = __half22float2(h[0]), b2 = __half22float2(h[1]), c2 = __half22float2(h[2]),
               d2 = __half22float2(h[3]);
        float sum = ((a.x + a.y) + (b2.x + b2.y)) + ((c2.x + c2.y) + (d2.x + d2.y));
        sum += __shfl_xor_sync(0xffffffffu, sum, 1);
        sum += __shfl_xor_sync(0xffffffffu, sum, 2);          // row 8n+g, whole block
        return sum;
      };
      float amax = 0.f;
#pragma unroll
      for (int bb = 0; bb < NB; ++bb) amax = fmaxf(amax, fabsf(block_sum(bb)));
      int qe = 0;                                   // |sum| <= 32 * 65504 < 2^21: qe <= 16
      while (qe < 16 && amax > ldexpf(32.f, qe)) ++qe;
      if (qe > 0) {
        const uint32_t down = pack_half2(ldexpf(1.f, -qe), ldexpf(1.f, -qe));   // exact power of two
#pragma unroll
        for (int bb = 0; bb < NB; ++bb) {
          qf[n][bb].x = hmul2_u32(qf[n][bb].x, down);
          qf[n][bb].y = hmul2_u32(qf[n][bb].y, down);
          qf[n][bb].z = hmul2_u32(qf[n][bb].z, down);
          qf[n][bb].w = hmul2_u32(qf[n][bb].w, down);
        }
      }
      // rows 2c and 2c + 1 of the score fragments are held by the lanes of g = 2c, 2c + 1
      row_scale[n][0] = ldexpf(p.scale_log2, __shfl_sync(0xffffffffu, qe, 8 * c));
      row_scale[n][1] = ldexpf(p.scale_log2, __shfl_sync(0xffffffffu, qe, 8 * c + 4));
      float csum[NB];
#pragma unroll
      for (int bb = 0; bb < NB; ++bb) csum[bb] = -1152.f * block_sum(bb);
      // B[k][row g]: thread (g, c) holds k = 2c, 2c+1 (b0b1) and 2c+8, 2c+9 (b2b3)
      uint32_t bw[2];
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        float v[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int k = 2 * c + 8 * half + e;
          const int blk = k % NB;
          const bool lo_part = (k / NB) == 1;
          float cv = 0.f;
#pragma unroll
          for (int bb = 0; bb < NB; ++bb) cv = (bb == blk) ? csum[bb] : cv;
          const float hi = __half2float(__float2half_rn(cv));
          v[e] = k < 2 * NB ? (lo_part ? cv - hi : hi) : 0.f;
        }
        bw[half] = pack_half2(v[0], v[1]);
      }
      corrb[n][0] = bw[0];
      corrb[n][1] = bw[1];
    }
  }

#pragma unroll
  for (int n = 0; n < NT; ++n) {
#pragma unroll
    for (int bb = 0; bb < NB; ++bb) {
      const uint4 v = qf[n][bb];
      if (!kSharedQFor<D> || warp == 0)
        asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(qsm + ((n * NB + bb) * 32 + lane) * 16), "r"(v.x),
                     "r"(v.y), "r"(v.z), "r"(v.w) : "memory");
    }
  }
  if constexpr (kSharedQFor<D>) __syncthreads();
  else __syncwarp();

  if (app_n > 0) {
    // Fused append: quantize this KV head's rows of the new tokens into their
    // pool pages (one row side per D/8 lanes, the same code as the append
    // kernel; even warps take the K rows and odd warps the V rows, so the two
    // sides run in parallel), then order those generic stores before the bulk
    // copies that read them.
    constexpr int kLanesRow = D / 8;
    constexpr int kRowsWarp = 32 / kLanesRow;
    constexpr int kRowsPass = (kWarps / 2) * kRowsWarp;
    const QuantTarget dst{const_cast<uint8_t *>(p.k_pool), const_cast<uint8_t *>(p.v_pool), p.n_kv_heads, KF, VF,
                          p.k_scale, p.v_scale};
    const int l = lane % kLanesRow;
    const bool v_side = warp & 1;            // warp-uniform
    const __half *src = v_side ? p.v_new : p.k_new;
    const int first_new = Tseq - p.q_len;    // position of new token 0
    for (int j0 = 0; j0 < app_n; j0 += kRowsPass) {
      const int j = j0 + (warp >> 1) * kRowsWarp + lane / kLanesRow;
      const int pos = app_pos0 + j;
      int page = -1;
      uint4 rx = make_uint4(0, 0, 0, 0);
      if (j < app_n) {
        page = pid_s[pos / kPage - tok0 / kPage];
        const size_t off = ((static_cast<size_t>(b) * p.q_len + (pos - first_new)) * p.n_kv_heads + kvh) * D + 8 * l;
        rx = *reinterpret_cast<const uint4 *>(src + off);
      }
      quantize_store_row<D>(dst, page >= 0, max(page, 0), pos % kPage, kvh, l, rx, rx, !v_side, v_side);
    }
    fence_proxy_async_global();
    __syncthreads();
    if (lane == 0) {
      for (int i = r; i < min(NS, npages); i += R)
        if (i >= app_lo && i <= app_hi) issue(i, i);
    }
  }

  float o[NT][2 * NB][4];
  float mt[NT][4];
  float mrow[NT][2], lrow[NT][2];
#pragma unroll
  for (int n = 0; n < NT; ++n) {
#pragma unroll
    for (int i = 0; i < 2 * NB; ++i) o[n][i][0] = o[n][i][1] = o[n][i][2] = o[n][i][3] = 0.f;
    mt[n][0] = mt[n][1] = mt[n][2] = mt[n][3] = 0.f;
    mrow[n][0] = mrow[n][1] = -INFINITY;
    lrow[n][0] = lrow[n][1] = 0.f;
  }

  int s = r, par = 0;            // stage and phase parity of page i
  int stop_at = -1;              // page whose wait gave up, if any
  for (int i = r; i < npages; i += R) {
    if (!mbar_wait_bounded(full0 + 8 * s, par, p.status, p.page_wait_ns)) {
      stop_at = i;
      break;
    }
    if (pid_s[i] >= 0) {
      // Pages wholly inside every row's visible range (all but the last one or
      // two of a sequence) take a path without any masking code.
      const int pos_first = tok0 + i * kPage;
      const bool plain = pos_first >= lo && pos_first + kPage <= T;
      auto page = [&](auto tail) {
        const uint32_t ka = ring + s * STAGE;
        const uint32_t va = ka + KSEG;
        const int pos0 = tok0 + i * kPage;
        constexpr bool masked = decltype(tail)::value;    // some key of the page is hidden from some row
        constexpr bool partial = decltype(tail)::value;   // the page runs past the sequence

        // ---------------------------------------------------- S^T = K^ Q^T --
        float sc[NT][4];
#pragma unroll
          for (int n = 0; n < NT; ++n) sc[n][0] = sc[n][1] = sc[n][2] = sc[n][3] = 0.f;
        if constexpr (kK4) {
          // NVFP4 K: the 8 codes of each A fragment in one word; each 16-element
          // block's e4m3 scale is folded into the fp16 codes (the product is exact)
          uint32_t kw[2 * NB];
#pragma unroll
          for (int q4 = 0; q4 < NB / 2; ++q4) {
            const uint4 x = lds128(ka + (q4 * 32 + lane) * 16);
            kw[4 * q4] = x.x; kw[4 * q4 + 1] = x.y; kw[4 * q4 + 2] = x.z; kw[4 * q4 + 3] = x.w;
          }
          // block scales of tokens g and g + 8, as fp16 pairs of blocks (2 bb, 2 bb + 1)
          uint32_t sg[NB], sg8[NB];
          {
            uint32_t wg[NB / 2], wg8[NB / 2];
            if constexpr (NB == 4) {
              const uint2 a = lds64(ka + 8 * D + g * 8), bq = lds64(ka + 8 * D + (g + 8) * 8);
              wg[0] = a.x; wg[1] = a.y; wg8[0] = bq.x; wg8[1] = bq.y;
            } else {
              const uint4 a = lds128(ka + 8 * D + g * 16), bq = lds128(ka + 8 * D + (g + 8) * 16);
              wg[0] = a.x; wg[1] = a.y; wg[2] = a.z; wg[3] = a.w;
              wg8[0] = bq.x; wg8[1] = bq.y; wg8[2] = bq.z; wg8[3] = bq.w;
            }
#pragma unroll
            for (int q2 = 0; q2 < NB / 2; ++q2) {
              e4m3x4_to_half2x2(wg[q2], sg[2 * q2], sg[2 * q2 + 1]);
              e4m3x4_to_half2x2(wg8[q2], sg8[2 * q2], sg8[2 * q2 + 1]);
            }
          }
          const uint32_t sel = c < 2 ? 0x1010u : 0x3232u;     // the thread's 8 dims lie in block 2 bb + c / 2
#pragma unroll
          for (int bb = 0; bb < NB; ++bb) {
            const uint32_t s0 = __byte_perm(sg[bb], 0u, sel), s1 = __byte_perm(sg8[bb], 0u, sel);
#pragma unroll
            for (int n = 0; n < NT; ++n) {
              const uint4 qv = lds128(qsm + ((n * NB + bb) * 32 + lane) * 16);
#pragma unroll
              for (int mm = 0; mm < 2; ++mm) {
                const uint32_t w = kw[2 * bb + mm];
                uint32_t a[4];
                e2m1x8_to_half2x4(w, a);
                a[0] = hmul2_u32(a[0], s0);           // token g
                a[1] = hmul2_u32(a[1], s1);           // token g + 8
                a[2] = hmul2_u32(a[2], s0);
                a[3] = hmul2_u32(a[3], s1);
                mma_16816(sc[n], a, mm == 0 ? qv.x : qv.z, mm == 0 ? qv.y : qv.w);
              }
            }
          }
        } else {
          uint4 kc[NB];
#pragma unroll
            for (int rr = 0; rr < NB; ++rr) kc[rr] = lds128(ka + (rr * 32 + lane) * 16);
          // q8_0 block scales of tokens g and g+8, two fp16 per word
          [[maybe_unused]] uint32_t dk0[NB / 2], dk1[NB / 2];
          if constexpr (kK8) {
            if constexpr (NB == 4) {
              const uint2 a = lds64(ka + 16 * D + g * NB * 2), bq = lds64(ka + 16 * D + (g + 8) * NB * 2);
              dk0[0] = a.x; dk0[1] = a.y; dk1[0] = bq.x; dk1[1] = bq.y;
            } else {
              const uint4 a = lds128(ka + 16 * D + g * NB * 2), bq = lds128(ka + 16 * D + (g + 8) * NB * 2);
              dk0[0] = a.x; dk0[1] = a.y; dk0[2] = a.z; dk0[3] = a.w;
              dk1[0] = bq.x; dk1[1] = bq.y; dk1[2] = bq.z; dk1[3] = bq.w;
            }
          }
#pragma unroll
            for (int bb = 0; bb < NB; ++bb) {
            const uint4 &c0 = kc[bb / 2];
            const uint4 &c1 = kc[NB / 2 + bb / 2];
            const uint32_t t0lo = (bb & 1) ? c0.z : c0.x, t0hi = (bb & 1) ? c0.w : c0.y;
            const uint32_t t1lo = (bb & 1) ? c1.z : c1.x, t1hi = (bb & 1) ? c1.w : c1.y;
            uint32_t a0[4], a1[4];
            k_pairs<KF>(t0lo, a0[0], a0[2]);
            k_pairs<KF>(t1lo, a0[1], a0[3]);
            k_pairs<KF>(t0hi, a1[0], a1[2]);
            k_pairs<KF>(t1hi, a1[1], a1[3]);
#pragma unroll
              for (int n = 0; n < NT; ++n) {
                const uint4 qv = lds128(qsm + ((n * NB + bb) * 32 + lane) * 16);
              if constexpr (kK8) {
                float acc[4] = {0.f, 0.f, 0.f, 0.f};
                mma_16816(acc, a0, qv.x, qv.y);
                mma_16816(acc, a1, qv.z, qv.w);
                const float2 dd0 = __half22float2(*reinterpret_cast<const __half2 *>(&dk0[bb / 2]));
                const float2 dd1 = __half22float2(*reinterpret_cast<const __half2 *>(&dk1[bb / 2]));
                const float d0 = (bb & 1) ? dd0.y : dd0.x, d1 = (bb & 1) ? dd1.y : dd1.x;
                sc[n][0] = fmaf(d0, acc[0], sc[n][0]);
                sc[n][1] = fmaf(d0, acc[1], sc[n][1]);
                sc[n][2] = fmaf(d1, acc[2], sc[n][2]);
                sc[n][3] = fmaf(d1, acc[3], sc[n][3]);
              } else {
                mma_16816(sc[n], a0, qv.x, qv.y);
                mma_16816(sc[n], a1, qv.z, qv.w);
              }
            }
          }
          if constexpr (kK8) {
            // bias removal: A[token][k] = d of block k % nb (k < 2nb), B = corrb
            uint32_t ad[4];
            if constexpr (NB == 4) {
              ad[0] = (c & 1) ? dk0[1] : dk0[0];
              ad[1] = (c & 1) ? dk1[1] : dk1[0];
              ad[2] = 0u;
              ad[3] = 0u;
            } else {
              const uint32_t x0 = c == 0 ? dk0[0] : c == 1 ? dk0[1] : c == 2 ? dk0[2] : dk0[3];
              const uint32_t x1 = c == 0 ? dk1[0] : c == 1 ? dk1[1] : c == 2 ? dk1[2] : dk1[3];
              ad[0] = x0;
              ad[1] = x1;
              ad[2] = x0;
              ad[3] = x1;
            }
#pragma unroll
              for (int n = 0; n < NT; ++n) mma_16816(sc[n], ad, corrb[n][0], corrb[n][1]);
          }
        }

        // ------------------------------------------------- online softmax --
        uint32_t pb[NT][2];
        float s4[NT][4];
        bool grow = false;      // some row's maximum passed its reference by more than kLazy
        float mx[NT][2];
#pragma unroll
          for (int n = 0; n < NT; ++n) {
          if constexpr (kK8) {
            s4[n][0] = sc[n][0] * row_scale[n][0];
            s4[n][1] = sc[n][1] * row_scale[n][1];
            s4[n][2] = sc[n][2] * row_scale[n][0];
            s4[n][3] = sc[n][3] * row_scale[n][1];
          } else {
#pragma unroll
            for (int e = 0; e < 4; ++e) s4[n][e] = sc[n][e] * p.scale_log2;
          }
          if (masked) {
            const int t0 = pos0 + g, t1 = pos0 + g + 8;
            const bool v0 = t0 < T && t0 >= lo, v1 = t1 < T && t1 >= lo;
            s4[n][0] = v0 ? s4[n][0] : -INFINITY;
            s4[n][1] = v0 ? s4[n][1] : -INFINITY;
            s4[n][2] = v1 ? s4[n][2] : -INFINITY;
            s4[n][3] = v1 ? s4[n][3] : -INFINITY;
          }
#pragma unroll
            for (int u = 0; u < 2; ++u) {
            float m1 = fmaxf(s4[n][u], s4[n][2 + u]);
            m1 = fmaxf(m1, __shfl_xor_sync(0xffffffffu, m1, 4));
            m1 = fmaxf(m1, __shfl_xor_sync(0xffffffffu, m1, 8));
            m1 = fmaxf(m1, __shfl_xor_sync(0xffffffffu, m1, 16));
            mx[n][u] = m1;
            grow = grow || (m1 > mrow[n][u] + kLazy);
          }
        }
        // The reference maximum of a row moves only when a score exceeds it by
        // more than kLazy (log2 units): until then the weights stay <= 4, and O
        // and l need no rescale.  4 keeps P * d (the V operand, d <= 65504/7)
        // finite in fp16 for any finite input.  Warp-uniform decision.
        if (__any_sync(0xffffffffu, grow)) {
#pragma unroll
            for (int n = 0; n < NT; ++n) {
#pragma unroll
              for (int u = 0; u < 2; ++u) {
              const float mnew = fmaxf(mrow[n][u], mx[n][u]);
              const float alpha = mnew == -INFINITY ? 1.f : fast_exp2(mrow[n][u] - mnew);
              mrow[n][u] = mnew;
              lrow[n][u] *= alpha;
#pragma unroll
                for (int i2 = 0; i2 < 2 * NB; ++i2) {
                o[n][i2][u] *= alpha;
                o[n][i2][2 + u] *= alpha;
              }
              if constexpr (kQ5) mt[n][u] *= alpha;
            }
          }
        }
#pragma unroll
          for (int n = 0; n < NT; ++n) {
          float p4[4];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
            const float muse = mrow[n][u] == -INFINITY ? 0.f : mrow[n][u];
            p4[u] = fast_exp2(s4[n][u] - muse);
            p4[2 + u] = fast_exp2(s4[n][2 + u] - muse);
            lrow[n][u] += p4[u] + p4[2 + u];
          }
          pb[n][0] = movmatrix_trans(pack_half2(p4[0], p4[1]));   // tokens 2c, 2c+1 of row g
          pb[n][1] = movmatrix_trans(pack_half2(p4[2], p4[3]));   // tokens 2c+8, 2c+9
        }

        // ---------------------------------------------- O^T += V^ P^T ---------
        // token-validity masks of the thread's B/A token pairs (partial pages only)
        uint32_t m01 = 0xFFFFFFFFu, m89 = 0xFFFFFFFFu;
        if (partial) {
          const int t = pos0 + 2 * c;
          auto vis = [&](int u) { return u < T && u >= lo; };
          m01 = (vis(t) ? 0x0000FFFFu : 0u) | (vis(t + 1) ? 0xFFFF0000u : 0u);
          m89 = (vis(t + 8) ? 0x0000FFFFu : 0u) | (vis(t + 9) ? 0xFFFF0000u : 0u);
        }
        if constexpr (kVq) {
          constexpr int DOFF = kQ5 ? 10 * D : 8 * D;
          uint2 dv[NB];
#pragma unroll
            for (int q2 = 0; q2 < NB / 2; ++q2) {
            const uint4 x = lds128(va + DOFF + c * NB * 8 + q2 * 16);
            dv[2 * q2] = make_uint2(x.x, x.y);
            dv[2 * q2 + 1] = make_uint2(x.z, x.w);
          }
          if (partial) {
#pragma unroll
              for (int bb = 0; bb < NB; ++bb) {
              dv[bb].x &= m01;
              dv[bb].y &= m89;
            }
          }
          [[maybe_unused]] uint32_t hw[NB / 2];
          if constexpr (kQ5) {
            if constexpr (NB == 4) {
              const uint2 x = lds64(va + 8 * D + lane * (NB / 2) * 4);
              hw[0] = x.x;
              hw[1] = x.y;
            } else {
              const uint4 x = lds128(va + 8 * D + lane * (NB / 2) * 4);
              hw[0] = x.x; hw[1] = x.y; hw[2] = x.z; hw[3] = x.w;
            }
          }
#pragma unroll
            for (int bp = 0; bp < NB / 2; ++bp) {
            const uint4 nw = lds128(va + (bp * 32 + lane) * 16);
#pragma unroll
              for (int bh = 0; bh < 2; ++bh) {
              const int bb = 2 * bp + bh;
              uint32_t bs[NT][2];
#pragma unroll
                for (int n = 0; n < NT; ++n) {
                bs[n][0] = hmul2_u32(pb[n][0], dv[bb].x);
                bs[n][1] = hmul2_u32(pb[n][1], dv[bb].y);
              }
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                const uint32_t w = bh == 0 ? (h == 0 ? nw.x : nw.y) : (h == 0 ? nw.z : nw.w);
                // Pairs 0 and 2 (dim slot g) become 1024 + code, pairs 1 and 3 (slot
                // g+8) 1024 + 16 code: nibbles spliced under the exponent of 1024,
                // the odd pairs without a shift.
                const uint32_t w8 = w >> 8;
                uint32_t a[4];
                a[0] = (w & 0x000F000Fu) | 0x64006400u;
                a[1] = (w & 0x00F000F0u) | 0x64006400u;
                a[2] = (w8 & 0x000F000Fu) | 0x64006400u;
                a[3] = (w8 & 0x00F000F0u) | 0x64006400u;
                if constexpr (kQ5) {
                  // bit 4 of the codes of nibble word k = 2*(bb%2) + h sits at
                  // 4s + 16f + k + 8p of the block pair's word: two shifts place
                  // it at 16 (pairs 0, 2) or 256 (pairs 1, 3) of the fp16 value.
                  const int k = 2 * bh + h;
                  const uint32_t x0 = hw[bp] << (4 - k);
                  const uint32_t x1 = (hw[bp] >> 8) << (4 - k);          // (H >> 8) << (4 - k) == H >> (4 + k) on the bits kept
                  a[0] |= x0 & 0x00100010u;
                  a[1] |= x0 & 0x01000100u;
                  a[2] |= x1 & 0x00100010u;
                  a[3] |= x1 & 0x01000100u;
                }
                // exact back to the code: x - 1024 (q4_0: - 1032), x / 16 - 64 (q4_0: - 72),
                // on the FMA pipe (the ALU pipe is the busier one)
                constexpr uint32_t kSub0 = kQ5 ? 0x64006400u : 0x64086408u;      // 1024 | 1032
                constexpr uint32_t kSub1 = kQ5 ? 0xD400D400u : 0xD480D480u;      // -64 | -72
                a[0] = hsub2_u32(a[0], kSub0);
                a[2] = hsub2_u32(a[2], kSub0);
                a[1] = hfma2_u32(a[1], 0x2C002C00u, kSub1);
                a[3] = hfma2_u32(a[3], 0x2C002C00u, kSub1);
#pragma unroll
                  for (int n = 0; n < NT; ++n) mma_16816(o[n][2 * bb + h], a, bs[n][0], bs[n][1]);
              }
            }
          }
          if constexpr (kQ5) {
            uint2 mv = make_uint2(0, 0);
            if (g < NB) {
              mv = lds64(va + 11 * D + (c * NB + g) * 8);
              if (partial) {
                mv.x &= m01;
                mv.y &= m89;
              }
            }
            const uint32_t am[4] = {mv.x, 0u, mv.y, 0u};
#pragma unroll
              for (int n = 0; n < NT; ++n) mma_16816(mt[n], am, pb[n][0], pb[n][1]);
          }
        } else if constexpr (kV4) {
          // NVFP4 V: m-tile i is 16-element block i (dims 16 i + g, 16 i + g + 8).
          // Each byte holds one token's codes of dims g and g + 8; two tokens'
          // bytes convert to fp16 pairs and are regrouped by token pair.  The
          // per-token block scale is folded into P (masked to 0 past the keys).
          uint32_t sw[2 * NB];
#pragma unroll
          for (int q4 = 0; q4 < NB / 2; ++q4) {
            const uint4 x = lds128(va + 8 * D + c * (2 * NB) * 4 + q4 * 16);
            sw[4 * q4] = x.x; sw[4 * q4 + 1] = x.y; sw[4 * q4 + 2] = x.z; sw[4 * q4 + 3] = x.w;
          }
#pragma unroll
          for (int q4 = 0; q4 < NB / 2; ++q4) {
            const uint4 cw = lds128(va + (q4 * 32 + lane) * 16);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const int i = 4 * q4 + u;
              const uint32_t w = u == 0 ? cw.x : u == 1 ? cw.y : u == 2 ? cw.z : cw.w;
              uint32_t s01, s89;
              e4m3x4_to_half2x2(sw[i], s01, s89);
              if (partial) {
                s01 &= m01;
                s89 &= m89;
              }
              uint32_t h[4];
              e2m1x8_to_half2x4(w, h);
              uint32_t a[4];
              a[0] = __byte_perm(h[0], h[1], 0x5410u);     // dim g: tokens 2c, 2c + 1
              a[1] = __byte_perm(h[0], h[1], 0x7632u);     // dim g + 8
              a[2] = __byte_perm(h[2], h[3], 0x5410u);     // tokens 2c + 8, 2c + 9
              a[3] = __byte_perm(h[2], h[3], 0x7632u);
#pragma unroll
              for (int n = 0; n < NT; ++n)
                mma_16816(o[n][i], a, hmul2_u32(pb[n][0], s01), hmul2_u32(pb[n][1], s89));
            }
          }
        } else {  // fp8 V
#pragma unroll
            for (int bb = 0; bb < NB; ++bb) {
            const uint4 x = lds128(va + (bb * 32 + lane) * 16);
#pragma unroll
              for (int h = 0; h < 2; ++h) {
              const uint32_t w0 = h == 0 ? x.x : x.z, w1 = h == 0 ? x.y : x.w;
              uint32_t a[4];
              e4m3x4_to_half2x2(w0, a[0], a[1]);
              e4m3x4_to_half2x2(w1, a[2], a[3]);
              if (partial) {
                a[0] &= m01; a[1] &= m01; a[2] &= m89; a[3] &= m89;
              }
#pragma unroll
                for (int n = 0; n < NT; ++n) mma_16816(o[n][2 * bb + h], a, pb[n][0], pb[n][1]);
            }
          }
        }
          };
      if (plain)
        page(std::false_type{});
      else
        page(std::true_type{});
    }
    __syncwarp();
    // The stage is read: refill it with page i + NS (this warp's next page there).
    if (lane == 0 && i + NS < npages) {
      fence_proxy_async();
      issue(i + NS, s);
    }
    s += R;
    if (s >= NS) {
      s -= NS;
      par ^= 1;
    }
  }
  // A wait that gave up: stay until this lane's copies in flight have landed,
  // so no bulk copy outlives the CTA's shared memory.  Each of those waits has
  // the full limit; a stage whose phase cannot complete (its expected bytes
  // were never all sent) costs one limit and holds no copy in flight, since a
  // copy's bytes land before they count against the phase.
  if (stop_at >= 0 && lane == 0) {
    for (int j = stop_at; j < min(stop_at + NS, npages); j += R)
      mbar_wait_bounded(full0 + 8 * (j % NS), (j / NS) & 1, p.status);
  }

  // ------------------------------------------------------ merge the warps --
#pragma unroll
  for (int n = 0; n < NT; ++n) {
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      float l = lrow[n][u];
      l += __shfl_xor_sync(0xffffffffu, l, 4);
      l += __shfl_xor_sync(0xffffffffu, l, 8);
      l += __shfl_xor_sync(0xffffffffu, l, 16);
      lrow[n][u] = l;
    }
  }
  __syncthreads();                       // every warp is done with the ring
  float *mo = reinterpret_cast<float *>(smem);
  float *mm = mo + ML::kO;
  float *ml = mm + ML::kM;
  float *mterm = ml + ML::kM;
#pragma unroll
  for (int n = 0; n < NT; ++n) {
    const int lr0 = warp * ROWS_W + 8 * n + 2 * c;
#pragma unroll
    for (int i = 0; i < 2 * NB; ++i) {
      // dims of m-tile i's rows g and g + 8 (the V layout's dim order)
      const int ja = kV4 ? 16 * i + g : 32 * (i / 2) + 4 * g + 2 * (i % 2);
      const int jb = kV4 ? ja + 8 : ja + 1;
      mo[lr0 * D + ja] = o[n][i][0];
      mo[(lr0 + 1) * D + ja] = o[n][i][1];
      mo[lr0 * D + jb] = o[n][i][2];
      mo[(lr0 + 1) * D + jb] = o[n][i][3];
    }
    if (g == 0) {
      mm[lr0] = mrow[n][0];
      mm[lr0 + 1] = mrow[n][1];
      ml[lr0] = lrow[n][0];
      ml[lr0 + 1] = lrow[n][1];
    }
    if constexpr (kQ5) {
      if (g < NB) {
        mterm[lr0 * NB + g] = mt[n][0];
        mterm[(lr0 + 1) * NB + g] = mt[n][1];
      }
    }
  }
  __syncthreads();

  const float vscale = p.v_scale;            // 1 unless V has a per-tensor scale
  for (int item = tid; item < nrows * (D / 4); item += kThreads) {
    const int lr = item / (D / 4);
    const int j4 = (item % (D / 4)) * 4;
    float M = -INFINITY;
    for (int rr = 0; rr < R; ++rr) M = fmaxf(M, mm[rr * ROWS_W + lr]);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float L = 0.f;
    if (M != -INFINITY) {
      for (int rr = 0; rr < R; ++rr) {
        const int wr = rr * ROWS_W + lr;
        const float wgt = fast_exp2(mm[wr] - M);
        L = fmaf(wgt, ml[wr], L);
        const float4 x = *reinterpret_cast<const float4 *>(mo + wr * D + j4);
        const float add = kQ5 ? mterm[wr * NB + j4 / 32] : 0.f;
        acc.x = fmaf(wgt, x.x + add, acc.x);
        acc.y = fmaf(wgt, x.y + add, acc.y);
        acc.z = fmaf(wgt, x.z + add, acc.z);
        acc.w = fmaf(wgt, x.w + add, acc.w);
      }
    }
    const float inv = L > 0.f ? vscale / L : 0.f;
    acc.x *= inv; acc.y *= inv; acc.z *= inv; acc.w *= inv;
    const int head = kvh * p.group + 8 * hg + lr;
    const size_t rowid = (static_cast<size_t>(b) * p.q_len + qi) * p.n_heads + head;
    if (nsplit_b == 1 && p.skip == 0) {
      uint2 h;
      h.x = pack_half2(acc.x, acc.y);
      h.y = pack_half2(acc.z, acc.w);
      *reinterpret_cast<uint2 *>(p.out + rowid * D + j4) = h;
    } else {
      const size_t pidx = rowid * p.nsplit_max + split;
      *reinterpret_cast<float4 *>(p.o_part + pidx * D + j4) = acc;
      if (j4 == 0) p.lse_part[pidx] = L > 0.f ? M + __log2f(L) : -INFINITY;
    }
  }
  if (waits_for_prefix) grid_dependency_wait();
}

// One dispatcher per translation unit (head_dim).
cudaError_t launch_decode_d128(int kf, int vf, const DecodeParams &p, dim3 grid, size_t smem, cudaStream_t st);
cudaError_t launch_decode_d256(int kf, int vf, const DecodeParams &p, dim3 grid, size_t smem, cudaStream_t st);

template <int D, int KF, int VF>
cudaError_t launch_one(const DecodeParams &p, dim3 grid, size_t smem, cudaStream_t st) {
  static bool configured = false;   // per instantiation; attribute is per device function
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(decode_split_kernel<D, KF, VF>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  return launch_pdl(decode_split_kernel<D, KF, VF>, grid, dim3(kWarpsFor<D> * 32), smem, st, p);
}

template <int D>
cudaError_t dispatch_formats(int kf, int vf, const DecodeParams &p, dim3 grid, size_t smem, cudaStream_t st) {
  auto by_v = [&](auto kc) -> cudaError_t {
    constexpr int K = decltype(kc)::value;
    switch (vf) {
      case MEMRA_KV_Q5_1: return launch_one<D, K, MEMRA_KV_Q5_1>(p, grid, smem, st);
      case MEMRA_KV_Q4_0: return launch_one<D, K, MEMRA_KV_Q4_0>(p, grid, smem, st);
      case MEMRA_KV_FP8_E4M3: return launch_one<D, K, MEMRA_KV_FP8_E4M3>(p, grid, smem, st);
      case MEMRA_KV_NVFP4: return launch_one<D, K, MEMRA_KV_NVFP4>(p, grid, smem, st);
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

}  // namespace memra
