// Quantize-and-store of one K/V row into the paged pools: the block rules
// and byte layout stated in include/memra.h, shared by the append kernel and
// by the decode kernel's fused append.  The rounding is exact in float32 (see
// kv_append.cu).
#pragma once

#include "memra_device.cuh"

namespace memra {

struct QuantTarget {
  uint8_t *k_pool;
  uint8_t *v_pool;
  int n_kv_heads, k_fmt, v_fmt;
  float k_scale, v_scale;
};

__device__ __forceinline__ float group4_max(float x) {
  x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, 1));
  return fmaxf(x, __shfl_xor_sync(0xffffffffu, x, 2));
}
__device__ __forceinline__ float group4_min(float x) {
  x = fminf(x, __shfl_xor_sync(0xffffffffu, x, 1));
  return fminf(x, __shfl_xor_sync(0xffffffffu, x, 2));
}

__device__ __forceinline__ void store_half(uint8_t *p, __half h) {
  *reinterpret_cast<__half *>(p) = h;
}

// a - b = hi + lo exactly (TwoSum of a and -b).
__device__ __forceinline__ void two_diff(float a, float b, float &hi, float &lo) {
  hi = __fsub_rn(a, b);
  const float bb = __fsub_rn(hi, a);
  lo = __fadd_rn(__fsub_rn(a, __fsub_rn(hi, bb)), __fsub_rn(-b, bb));
}

// fp16 round-to-nearest-even of (hi + lo) / k for hi + lo >= 0 and k in {7, 31, 127}.
// The candidate is the fp16 rounding of hi * fp32(1/k): within one fp16 step
// of the answer, since hi * fp32(1/k) is within 2^-22 (relative) of the
// quotient.  The sign of (hi + lo) / k minus each neighbouring midpoint then
// decides one step up or down, exactly: k times an fp16 midpoint has at most
// 19 significant bits, and hi minus it is exact by Sterbenz's lemma.  No
// branches: a warp's lanes never diverge here.
__device__ __forceinline__ __half fp16_quotient_rne(float hi, float lo, float k) {
  const float inv_k = k == 127.f ? 1.f / 127.f : (k == 31.f ? 1.f / 31.f : 1.f / 7.f);
  const unsigned hb = __half_as_ushort(__float2half_rn(__fmul_rn(hi, inv_k)));
  const float v = __half2float(__ushort_as_half(static_cast<unsigned short>(hb)));
  const float up_mid = 0.5f * (v + __half2float(__ushort_as_half(static_cast<unsigned short>(hb + 1))));
  const float dn_mid = 0.5f * (v + __half2float(__ushort_as_half(static_cast<unsigned short>(hb > 0 ? hb - 1 : 0))));
  const float t_up = __fadd_rn(__fsub_rn(hi, __fmul_rn(k, up_mid)), lo);     // sign of x/k - up_mid
  const float t_dn = __fadd_rn(__fsub_rn(hi, __fmul_rn(k, dn_mid)), lo);     // sign of x/k - dn_mid
  const bool odd = hb & 1u;
  const bool up = t_up > 0.f || (t_up == 0.f && odd);
  const bool dn = !up && hb > 0 && (t_dn < 0.f || (t_dn == 0.f && odd));
  return __ushort_as_half(static_cast<unsigned short>(hb + (up ? 1 : 0) - (dn ? 1 : 0)));
}

// Reciprocal of a block scale for quant_code's candidate (any value within a
// few ulps of 1/d serves; 1 for d == 0, whose codes are 0).
__device__ __forceinline__ float scale_reciprocal(float d) { return __fdividef(1.f, d == 0.f ? 1.f : d); }

// clamp(rne((hi + lo) / d), lo_q, hi_q) for the stored fp16 d (as float); 0 when d == 0.
// rd = scale_reciprocal(d).  The candidate is hi * rd rounded to the nearest
// integer by adding 1.5 * 2^23 (float32 rounding is to nearest even, and the
// integer then sits in the low mantissa bits): within one of the answer,
// since |hi / d| < 2^8.  q0 * d is exact (8 + 11 significant bits) and so is
// hi - q0 * d (Sterbenz); the signs of x/d - (q0 +- 1/2) then pick the code,
// ties to even.  No branches.
__device__ __forceinline__ int quant_code(float hi, float lo, float d, float rd, int lo_q, int hi_q) {
  constexpr float kRound = 12582912.f;                           // 1.5 * 2^23
  const float t = __fadd_rn(__fmul_rn(hi, rd), kRound);
  int q = __float_as_int(t) - __float_as_int(kRound);
  const float q0 = __fsub_rn(t, kRound);                         // exact
  const float e = __fsub_rn(hi, __fmul_rn(q0, d));               // exact
  const float hd = 0.5f * d;
  const float up = __fadd_rn(__fsub_rn(e, hd), lo);              // sign of x/d - (q0 + 1/2)
  const float dn = __fadd_rn(__fadd_rn(e, hd), lo);              // sign of x/d - (q0 - 1/2)
  // Sign tests on the bits (a float is > 0 iff its bits are > 0 as an int, and
  // zero iff they are 0 after the sign bit): fewer predicates than float
  // compares, so the eight codes of a lane interleave.  Up and down never both
  // hold (dn exceeds up by d).
  const int iu = __float_as_int(up), id = __float_as_int(dn), odd = q & 1;
  const int zu = (iu << 1) == 0, zd = (id << 1) == 0;
  q += ((iu > 0) | (zu & odd)) - (((id < 0) & !zd) | (zd & odd));
  return d == 0.f ? 0 : min(max(q, lo_q), hi_q);
}

// The IEEE float32 quotient RN(x / s) of an fp16 value x by a scale s, given
// r = RN(1 / s), without a division: x * r is within two ulps of the
// quotient, one refinement q + RN(x - q s) r brings it within one ulp, and a
// second gives the correctly rounded quotient (Markstein's division
// theorem: the remainder of a quotient within one ulp is exact, and
// RN(q + (x - q s) r) = RN(x / s) for r = RN(1 / s)).  The fp8 and NVFP4
// rules round this quotient, so it must be the IEEE one: a GPU test checks
// it against __fdiv_rn for every finite fp16 x over thousands of scales.
// Scales outside [2^-60, 2^60], where a remainder could leave the normal
// range, take the IEEE division.  A warp spends ~200 cycles on each IEEE
// division, a few on this.
__device__ __forceinline__ float div_by_scale(float x, float s, float r) {
  if (!(s >= 0x1p-60f && s <= 0x1p60f)) return __fdiv_rn(x, s);
  const float q0 = __fmul_rn(x, r);
  const float q1 = __fmaf_rn(__fmaf_rn(-q0, s, x), r, q0);
  const float q2 = __fmaf_rn(__fmaf_rn(-q1, s, x), r, q1);
  return x == 0.f ? q0 : q2;        // a zero keeps its sign
}

// NVFP4 codes of this lane's 8 elements (one half of a 16-element block; the
// partner half is on lane l ^ 1): e4m3 block scale of max|x| / (6 s) and E2M1
// codes of x / (scale * s), each step one float32 operation.  Returns the
// scale byte; codes[i] holds element i's 4-bit code.
__device__ __forceinline__ uint32_t nvfp4_half_block(const float (&x)[8], float s, uint32_t (&codes)[8]) {
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(x[i]));
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
  const float s6 = __fmul_rn(6.f, s);
  const float u = div_by_scale(amax, s6, __frcp_rn(s6));
  const uint32_t sb = __nv_cvt_float_to_fp8(u, __NV_SATFINITE, __NV_E4M3);
  const float eff = __fmul_rn(__half2float(__half(__nv_cvt_fp8_to_halfraw(static_cast<__nv_fp8_storage_t>(sb),
                                                                              __NV_E4M3))), s);
  const float reff = __frcp_rn(sb != 0 ? eff : 1.f);
#pragma unroll
  for (int i = 0; i < 8; i += 2) {
    uint32_t two = 0;
    if (sb != 0) two = float2_to_e2m1x2(div_by_scale(x[i + 1], eff, reff), div_by_scale(x[i], eff, reff));
    codes[i] = two & 0xFu;
    codes[i + 1] = two >> 4;
  }
  return sb;
}

// One (token, KV head) row per group of D/8 consecutive lanes; lane l of the
// group holds elements 8l..8l+7 of the K row (rk) and of the V row (rv).
// Every lane of the warp must call it, with the same do_k / do_v (it shuffles
// within the group); only rows with act set are stored, at token t of pool
// page `page`.  do_k / do_v select the sides to quantize (a caller may give K
// and V of a row to different warps, which then run in parallel).
template <int D>
__device__ __forceinline__ void quantize_store_row(const QuantTarget &dst, bool act, int page, int t, int head,
                                                   int l, uint4 rk, uint4 rv, bool do_k = true,
                                                   bool do_v = true) {
  constexpr int kNb = D / 32;
  const int b = l / 4;                            // block
  const int cc = l % 4;                           // 8-element chunk within the block
  // Both K and V of the row; shuffles below run on every lane (inactive rows
  // carry zeros), stores only on active rows.
  float xk[8], xv[8];
  {
    if (!act) {
      rk = make_uint4(0, 0, 0, 0);
      rv = make_uint4(0, 0, 0, 0);
    }
    const __half2 *hk = reinterpret_cast<const __half2 *>(&rk);
    const __half2 *hv = reinterpret_cast<const __half2 *>(&rv);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float2 a = __half22float2(hk[i]);
      float2 c = __half22float2(hv[i]);
      xk[2 * i] = a.x; xk[2 * i + 1] = a.y;
      xv[2 * i] = c.x; xv[2 * i + 1] = c.y;
    }
  }

  // ------------------------------------------------------------------ K ---
  if (!do_k) {
  } else if (dst.k_fmt == MEMRA_KV_NVFP4) {
    uint8_t *seg = dst.k_pool + (static_cast<size_t>(page) * dst.n_kv_heads + head) * k_seg_bytes(dst.k_fmt, D);
    uint32_t code[8];
    const uint32_t sb = nvfp4_half_block(xk, dst.k_scale, code);
    // this lane holds elements 8 l .. 8 l + 7: c = l % 4 of 32-element block l / 4, in 16-block l / 2
    const int lane_k = 4 * (t % 8) + l % 4;
    if (act) {
#pragma unroll
      for (int e = 0; e < 8; e += 2) {       // elements e, e + 1 share a byte
        const int w = 2 * (l / 4) + e / 4;
        seg[((w / 4) * 32 + lane_k) * 16 + (w % 4) * 4 + t / 8 + 2 * ((e % 4) / 2)] =
            static_cast<uint8_t>(code[e] | (code[e + 1] << 4));
      }
      if (l % 2 == 0) seg[8 * D + t * (D / 16) + l / 2] = static_cast<uint8_t>(sb);
    }
  } else {
    uint8_t *seg = dst.k_pool + (static_cast<size_t>(page) * dst.n_kv_heads + head) * k_seg_bytes(dst.k_fmt, D);
    const int tg = t % 8, tp = t / 8;
    const int chunk = (tp * (kNb / 2) + b / 2) * 32 + 4 * tg + cc;
    uint8_t code[8];
    if (dst.k_fmt == MEMRA_KV_Q8_0) {
      float amax = 0.f;
#pragma unroll
      for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(xk[i]));
      amax = group4_max(amax);
      const __half dh = fp16_quotient_rne(amax, 0.f, 127.f);
      const float d = __half2float(dh), rd = scale_reciprocal(d);
#pragma unroll
      for (int i = 0; i < 8; ++i)
        code[i] = static_cast<uint8_t>(quant_code(xk[i], 0.f, d, rd, -127, 127) + 128);   // stored biased
      if (act && cc == 0) store_half(seg + 16 * D + (t * kNb + b) * 2, dh);
    } else {
      const float r = __frcp_rn(dst.k_scale);
#pragma unroll
      for (int i = 0; i < 8; ++i)
        code[i] = __nv_cvt_float_to_fp8(div_by_scale(xk[i], dst.k_scale, r), __NV_SATFINITE, __NV_E4M3);
    }
    if (act) {
      uint2 w;
      w.x = code[0] | (code[1] << 8) | (code[2] << 16) | (static_cast<uint32_t>(code[3]) << 24);
      w.y = code[4] | (code[5] << 8) | (code[6] << 16) | (static_cast<uint32_t>(code[7]) << 24);
      *reinterpret_cast<uint2 *>(seg + chunk * 16 + (b % 2) * 8) = w;
    }
  }

  // ------------------------------------------------------------------ V ---
  if (!do_v) {
  } else if (dst.v_fmt == MEMRA_KV_NVFP4) {
    uint8_t *seg = dst.v_pool + (static_cast<size_t>(page) * dst.n_kv_heads + head) * v_seg_bytes(dst.v_fmt, D);
    uint32_t code[8];
    const uint32_t sb = nvfp4_half_block(xv, dst.v_scale, code);
    const int b16 = l / 2, vh = l % 2;     // this lane holds elements r = 8 vh .. 8 vh + 7 of block b16
    // elements r and r + 8 of the block share a byte: the even lane gathers its partner's codes
    uint32_t mine = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) mine |= code[i] << (4 * i);
    const uint32_t other = __shfl_xor_sync(0xffffffffu, mine, 1);
    const int c = (t % 8) / 2;
    if (act && vh == 0) {
#pragma unroll
      for (int r = 0; r < 8; ++r) {
        const int lane_v = 4 * r + c;
        seg[((b16 / 4) * 32 + lane_v) * 16 + (b16 % 4) * 4 + t % 2 + 2 * (t / 8)] =
            static_cast<uint8_t>(code[r] | (((other >> (4 * r)) & 0xFu) << 4));
      }
      seg[8 * D + (c * (D / 16) + b16) * 4 + t % 2 + 2 * (t / 8)] = static_cast<uint8_t>(sb);
    }
  } else {
    uint8_t *seg = dst.v_pool + (static_cast<size_t>(page) * dst.n_kv_heads + head) * v_seg_bytes(dst.v_fmt, D);
    const int c = (t % 8) / 2, f = t % 2, pp = t / 8, k = 2 * f + pp;
    // element i of this lane: r = 8*cc + i -> vg = 2*cc + i/4, h = (i%4)/2, s = i%2
    if (dst.v_fmt == MEMRA_KV_FP8_E4M3) {
      if (act) {
        const float r = __frcp_rn(dst.v_scale);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int vg = 2 * cc + i / 4, h = (i % 4) / 2, s = i % 2;
          const uint8_t byte = __nv_cvt_float_to_fp8(div_by_scale(xv[i], dst.v_scale, r), __NV_SATFINITE, __NV_E4M3);
          seg[(b * 32 + 4 * vg + c) * 16 + 8 * h + 2 * (2 * pp + s) + f] = byte;
        }
      }
    } else {
      int q[8];
      __half dh, mh = __float2half(0.f);
      if (dst.v_fmt == MEMRA_KV_Q5_1) {
        float mn = xv[0], mx = xv[0];
#pragma unroll
        for (int i = 1; i < 8; ++i) { mn = fminf(mn, xv[i]); mx = fmaxf(mx, xv[i]); }
        mn = group4_min(mn);
        mx = group4_max(mx);
        float rh, rl;
        two_diff(mx, mn, rh, rl);
        dh = fp16_quotient_rne(rh, rl, 31.f);
        mh = __float2half_rn(mn);                      // exact: mn is an fp16 value
        const float d = __half2float(dh), rd = scale_reciprocal(d);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          float xh, xl;
          two_diff(xv[i], mn, xh, xl);
          q[i] = quant_code(xh, xl, d, rd, 0, 31);
        }
      } else {  // q4_0, nibble = q + 8
        float amax = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(xv[i]));
        amax = group4_max(amax);
        dh = fp16_quotient_rne(amax, 0.f, 7.f);
        const float d = __half2float(dh), rd = scale_reciprocal(d);
#pragma unroll
        for (int i = 0; i < 8; ++i) q[i] = quant_code(xv[i], 0.f, d, rd, -8, 7) + 8;
      }
      // low nibbles: one byte per (vg, h) holding s = 0 (low) and s = 1 (high)
      if (act) {
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const int vg = 2 * cc + u;
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int i0 = 4 * u + 2 * h;
            const uint8_t byte = static_cast<uint8_t>((q[i0] & 15) | ((q[i0 + 1] & 15) << 4));
            seg[((b / 2) * 32 + 4 * vg + c) * 16 + (b % 2) * 8 + 4 * h + k] = byte;
          }
        }
      }
      if (dst.v_fmt == MEMRA_KV_Q5_1) {
        // bit 4 of each code: the byte of (vg, token) holds bit 4*s + 2*(b%2) + h,
        // so the even block's lane merges its partner's bits (shifted by 2).
        uint32_t hn[2];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          hn[u] = 0;
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int h = e / 2, s = e % 2;
            hn[u] |= static_cast<uint32_t>((q[4 * u + e] >> 4) & 1) << (4 * s + h);
          }
        }
        const uint32_t mine = hn[0] | (hn[1] << 8);
        const uint32_t other = __shfl_xor_sync(0xffffffffu, mine, 4);   // lane of block b^1
        if (act && (b % 2) == 0) {
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const int vg = 2 * cc + u;
            const uint32_t lo = (mine >> (8 * u)) & 0x33u, hi = (other >> (8 * u)) & 0x33u;
            seg[8 * D + ((4 * vg + c) * (kNb / 2) + b / 2) * 4 + k] = static_cast<uint8_t>(lo | (hi << 2));
          }
        }
      }
      if (act && cc == 0) {
        const int poff = ((c * kNb + b) * 4 + 2 * pp + f) * 2;
        if (dst.v_fmt == MEMRA_KV_Q5_1) {
          store_half(seg + 10 * D + poff, dh);
          store_half(seg + 11 * D + poff, mh);
        } else {
          store_half(seg + 8 * D + poff, dh);
        }
      }
    }
  }
}

}  // namespace memra
