// Device helpers shared by the library's kernels: hand-written PTX for
// mbarriers, bulk copies (TMA, non-tensor form), warp-level tensor-core MMA
// and register transposes, plus the page layout constants of memra.h.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <cuda_fp8.h>
#include <stdint.h>

#include "../../include/memra.h"

namespace memra {

constexpr int kPage = MEMRA_PAGE_SIZE;
constexpr int kSplitTokens = MEMRA_SPLIT_TOKENS;            // smallest split
constexpr int kSplitTokensMax = MEMRA_SPLIT_TOKENS_MAX;      // largest split
constexpr int kSplitPagesMax = kSplitTokensMax / kPage;
// Smallest split of a cascade call's own keys (the part after the shared
// prefix): short, so that the few own keys of many sequences spread over the
// GPU, yet few enough CTAs that they run on the SMs the prefix pass leaves
// free, beside it.
constexpr int kCascadeSplitTokens = 512;

// Split size of a range of T tokens: enough splits to give one long sequence
// `target` CTAs per KV head, never below `min_tokens` (MEMRA_SPLIT_TOKENS; 512
// for a cascade call's own keys) or above 8192 tokens, a multiple of the page.  Depends on T
// and the device only.
__host__ __device__ __forceinline__ int split_tokens(int T, int target, int min_tokens) {
  const int t = target > 0 ? target : 1;
  int c = (T + t - 1) / t;
  c = (c + kPage - 1) / kPage * kPage;
  return c < min_tokens ? min_tokens : (c > kSplitTokensMax ? kSplitTokensMax : c);
}

// Segment bytes per (format, side, head_dim); see the layout in memra.h.
__host__ __device__ constexpr int k_seg_bytes(int fmt, int D) {
  return fmt == MEMRA_KV_Q8_0 ? 17 * D : fmt == MEMRA_KV_FP8_E4M3 ? 16 * D : fmt == MEMRA_KV_NVFP4 ? 9 * D : 0;
}
__host__ __device__ constexpr int v_seg_bytes(int fmt, int D) {
  return fmt == MEMRA_KV_Q5_1 ? 12 * D
       : fmt == MEMRA_KV_Q4_0 ? 9 * D
       : fmt == MEMRA_KV_FP8_E4M3 ? 16 * D
       : fmt == MEMRA_KV_NVFP4 ? 9 * D : 0;
}

// Bound on every pipeline wait: past it the kernel flags MEMRA_DEVERR_TIMEOUT
// and stops waiting, so a lost copy can never hang the GPU.
constexpr unsigned long long kWaitLimitNs = 1000000000ull;

__device__ __forceinline__ void flag_error(int *status, int bit) {
  if (status) atomicOr(status, bit);
}

__device__ __forceinline__ unsigned long long global_timer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ----------------------------------------------------------------- mbarrier --

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\t"
      "mbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(bar)
      : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\t"
      "mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(bar),
      "r"(bytes)
      : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Waits for the phase with the given parity to complete; gives up after
// limit_ns (kWaitLimitNs unless a test shortens it), flags
// MEMRA_DEVERR_TIMEOUT and returns false.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity, int *status,
                                                  unsigned long long limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_timer_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (global_timer_ns() - t0 > limit_ns) {
      flag_error(status, MEMRA_DEVERR_TIMEOUT);
      return false;
    }
  }
}

// 1-D bulk copy global -> shared completing on an mbarrier (TMA, no tensor
// map).  Both addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_copy_g2s(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar,
                                              uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar), "l"(policy)
      : "memory");
}

// The same without an L2 hint: data that other CTAs read again.
__device__ __forceinline__ void bulk_copy_g2s_nohint(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}

__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// Orders this thread's earlier generic-proxy shared-memory accesses before its
// later async-proxy (bulk copy) accesses of the same memory.
__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Orders this thread's generic-proxy global stores before later async-proxy
// (bulk copy) reads of the same bytes.
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

__device__ __forceinline__ void named_barrier_sync(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// ------------------------------------------------------------ tensor cores --

// D = A * B + C, m16n8k16, fp16 inputs, fp32 accumulators (warp-wide).
__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Transpose of an 8x8 b16 tile held in the m8n8 fragment layout.
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&h);
}

__device__ __forceinline__ uint32_t hmul2_u32(uint32_t a, uint32_t b) {
  __half2 r = __hmul2(*reinterpret_cast<__half2 *>(&a), *reinterpret_cast<__half2 *>(&b));
  return *reinterpret_cast<uint32_t *>(&r);
}

__device__ __forceinline__ uint32_t hfma2_u32(uint32_t a, uint32_t b, uint32_t c) {
  __half2 r = __hfma2(*reinterpret_cast<__half2 *>(&a), *reinterpret_cast<__half2 *>(&b),
                      *reinterpret_cast<__half2 *>(&c));
  return *reinterpret_cast<uint32_t *>(&r);
}

__device__ __forceinline__ uint32_t hsub2_u32(uint32_t a, uint32_t b) {
  __half2 r = __hsub2(*reinterpret_cast<__half2 *>(&a), *reinterpret_cast<__half2 *>(&b));
  return *reinterpret_cast<uint32_t *>(&r);
}

// Two e4m3 bytes (low byte -> low half) to an fp16 pair; exact.
__device__ __forceinline__ uint32_t e4m3x2_to_half2(uint32_t two_bytes) {
  __half2_raw r = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(two_bytes & 0xFFFFu), __NV_E4M3);
  return static_cast<uint32_t>(r.x) | (static_cast<uint32_t>(r.y) << 16);
}

// Two OCP E2M1 codes (bits 3..0 and 7..4 of `byte`) -> fp16x2 (low code in the low half).
__device__ __forceinline__ uint32_t e2m1x2_to_half2(uint32_t byte) {
  uint32_t r;
  asm("{\n\t.reg .b8 t;\n\tcvt.u8.u32 t, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, t;\n\t}" : "=r"(r) : "r"(byte));
  return r;
}

// Both byte pairs of `w` (four e4m3 codes) -> two fp16x2: bytes 0-1 into lo,
// bytes 2-3 into hi, split with one vector move.
__device__ __forceinline__ void e4m3x4_to_half2x2(uint32_t w, uint32_t &lo, uint32_t &hi) {
  asm("{\n\t.reg .b16 a, b;\n\tmov.b32 {a, b}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, a;\n\tcvt.rn.f16x2.e4m3x2 %1, b;\n\t}"
      : "=r"(lo), "=r"(hi) : "r"(w));
}

// All four bytes of `w` (eight E2M1 codes) -> four fp16x2, byte k into h[k].
// The bytes are split with one vector move, so no shift is needed per byte.
__device__ __forceinline__ void e2m1x8_to_half2x4(uint32_t w, uint32_t (&h)[4]) {
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\tcvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\tcvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
      : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3]) : "r"(w));
}

// E2M1 codes of two floats, round to nearest even, saturating at +-6: `hi`'s
// code in bits 7..4, `lo`'s in bits 3..0.
__device__ __forceinline__ uint32_t float2_to_e2m1x2(float hi, float lo) {
  uint32_t r;
  asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\tcvt.u32.u8 %0, t;\n\t}"
      : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}

__device__ __forceinline__ uint2 lds64(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
  return v;
}

// Programmatic dependent launch: wait for the grids this one depends on
// (complete, memory visible), and let the next grid in the stream launch.
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void allow_dependent_launch() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Launch with the programmatic-stream-serialization attribute, so the kernel
// may start while the previous kernel of the stream finishes; the kernel
// itself calls grid_dependency_wait() before touching anything that kernel
// may write.
template <typename Kernel, typename... Args>
__host__ cudaError_t launch_pdl(Kernel kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t st, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

}  // namespace memra
