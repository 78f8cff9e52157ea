// K1: quantize-append of fp16 K/V rows into the block-quantized paged pools.
//
// Formats and rules: memra-bench card, "drafts/kf4/ - archived experiment"
// (KV knobs K = q8_0 | fp8, V = q5_1 | q4_0 | fp8); the block rules and the
// byte layout are the ones stated in include/memra.h.
//
// One group of D/8 lanes handles one (token, kv-head) row: each lane loads 8
// consecutive fp16 elements with one 128-bit load (a 32-element block is four
// lanes), block max/min come from two xor-shuffles, and the codes go straight
// to the positions the decode kernel's fragments read.
//
// The rules round exact real quotients, so the arithmetic is exact in float32
// (GB300's float64 rate is far too low for a hot path): x - m is carried as an
// unevaluated pair hi + lo (Knuth's TwoSum), a candidate rounding comes from
// a multiplication by the divisor's reciprocal (no IEEE division: a warp
// spends ~200 cycles on each), and the candidate is then confirmed or moved by one
// step by testing the sign of (hi - k*mid) + lo against the neighbouring
// rounding midpoints mid, where k*mid and hi - k*mid are exact (few
// significant bits; Sterbenz's lemma) and the final addition keeps the sign of
// the exact sum.  Ties go to the even neighbour.
#include <cuda_runtime.h>

#include "kv_quant.cuh"

namespace memra {

struct AppendParams {
  const __half *k;
  const __half *v;
  const int32_t *slots;
  uint8_t *k_pool;
  uint8_t *v_pool;
  int32_t *status;
  int n_tok, n_kv_heads, num_pages, k_fmt, v_fmt;
  float k_scale, v_scale;
};

template <int D>
__global__ void __launch_bounds__(256) kv_append_kernel(AppendParams p) {
  const QuantTarget dst{p.k_pool, p.v_pool, p.n_kv_heads, p.k_fmt, p.v_fmt, p.k_scale, p.v_scale};
  constexpr int kLanesPerRow = D / 8;
  grid_dependency_wait();        // k / v may come from the kernel before this one
  allow_dependent_launch();      // the decode kernel may start its prologue
  const int gtid = blockIdx.x * blockDim.x + threadIdx.x;
  const int row = gtid / kLanesPerRow;            // (token, kv-head)
  const int l = gtid % kLanesPerRow;              // lane within the row
  const bool live = row < p.n_tok * p.n_kv_heads;
  const int tok = live ? row / p.n_kv_heads : 0;
  const int head = live ? row % p.n_kv_heads : 0;
  // The slot and the row's K/V are loaded together (one memory round trip).
  int slot = -1;
  uint4 rk = make_uint4(0, 0, 0, 0), rv = make_uint4(0, 0, 0, 0);
  if (live) {
    const size_t off = (static_cast<size_t>(tok) * p.n_kv_heads + head) * D + 8 * l;
    slot = p.slots[tok];
    rk = *reinterpret_cast<const uint4 *>(p.k + off);
    rv = *reinterpret_cast<const uint4 *>(p.v + off);
  }
  if (slot >= p.num_pages * kPage) {
    if (l == 0) flag_error(p.status, MEMRA_DEVERR_BAD_SLOT);
    slot = -1;
  }
  const bool act = live && slot >= 0;
  const int page = act ? slot / kPage : 0;
  const int t = act ? slot % kPage : 0;
  quantize_store_row<D>(dst, act, page, t, head, l, rk, rv);
}

cudaError_t launch_kv_append(const memra_kv_cache &c, const void *k, const void *v, const int32_t *slots, int n_tok,
                             cudaStream_t stream) {
  AppendParams p;
  p.k = static_cast<const __half *>(k);
  p.v = static_cast<const __half *>(v);
  p.slots = slots;
  p.k_pool = static_cast<uint8_t *>(c.k_pool);
  p.v_pool = static_cast<uint8_t *>(c.v_pool);
  p.status = c.status;
  p.n_tok = n_tok;
  p.n_kv_heads = c.n_kv_heads;
  p.num_pages = c.num_pages;
  p.k_fmt = c.k_fmt;
  p.v_fmt = c.v_fmt;
  p.k_scale = c.k_scale;
  p.v_scale = c.v_scale;
  const long long rows = static_cast<long long>(n_tok) * c.n_kv_heads;
  const long long threads = rows * (c.head_dim / 8);
  const int block = 256;
  const unsigned grid = static_cast<unsigned>((threads + block - 1) / block);
  if (c.head_dim == 128) return launch_pdl(kv_append_kernel<128>, dim3(grid), dim3(block), 0, stream, p);
  return launch_pdl(kv_append_kernel<256>, dim3(grid), dim3(block), 0, stream, p);
}

}  // namespace memra
