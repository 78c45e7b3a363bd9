// Softmax building blocks of the tensor-core prefill kernels, 64 score
// columns of one row at a time: column masks decided once per tile and warp,
// the row extreme of the raw scores, and the exponentials with their row sum
// and the 16-bit packing of P (packed_varlen_attention.rs, stages 2-4,
// streamed as an online softmax).
#pragma once

#include "pva_device.cuh"

namespace pva {

__device__ __forceinline__ float col_val(const uint32_t (&va)[32], const uint32_t (&vb)[32],
                                         int e) {
  return __uint_as_float(e < 32 ? va[e] : vb[e - 32]);
}

// Column masks, chosen once per tile and warp: kMaskNone (every column
// visible), kMaskHi (visible iff col < hi_c: the causal diagonal, where no row
// of the warp starts inside the tile) and kMaskBoth (lo_c <= col < hi_c, one
// unsigned compare).  The column is a compile-time constant in the unrolled
// loops, so a test is one integer compare and one select.
constexpr int kMaskNone = 0, kMaskHi = 1, kMaskBoth = 2, kHalfEmpty = 3;
template <int MASK>
__device__ __forceinline__ bool col_visible(int col, int lo_c, int hi_c, unsigned span) {
  if (MASK == kMaskNone) return true;
  if (MASK == kMaskHi) return col < hi_c;
  return (unsigned)(col - lo_c) < span;
}

// Extreme (max if UP, else min) of the raw scores of columns [c, c+64);
// a mask replaces the invisible columns by the neutral value.
template <bool UP, int MASK>
__device__ __forceinline__ float extreme64(const uint32_t (&va)[32], const uint32_t (&vb)[32],
                                           int c, int lo_c, int hi_c, float ext) {
  const float neutral = UP ? __int_as_float(0xff800000) : __int_as_float(0x7f800000);
  const unsigned span = hi_c > lo_c ? (unsigned)(hi_c - lo_c) : 0u;
  // four independent partial extremes: no 32-long dependency chain
  float acc[4] = {ext, neutral, neutral, neutral};
#pragma unroll
  for (int e = 0; e < 64; e += 2) {
    float x0 = col_val(va, vb, e), x1 = col_val(va, vb, e + 1);
    if (MASK != kMaskNone) {
      x0 = col_visible<MASK>(c + e, lo_c, hi_c, span) ? x0 : neutral;
      x1 = col_visible<MASK>(c + e + 1, lo_c, hi_c, span) ? x1 : neutral;
    }
    float& a = acc[(e >> 1) & 3];
    a = UP ? fmax3f(a, x0, x1) : fmin3f(a, x0, x1);
  }
  return UP ? fmaxf(fmax3f(acc[0], acc[1], acc[2]), acc[3])
            : fminf(fmin3f(acc[0], acc[1], acc[2]), acc[3]);
}

// p = 2^(x - m) for columns [c, c+64), x the transformed score; row sums in
// rs; p packed as 16-bit pairs into pw.  Each group of 16 columns is done in
// sweeps -- all exponents, then all ex2, then sums and packing -- so that 16
// independent ex2 are issued back to back rather than each waiting for the
// one before it.
template <typename T, bool CAP, int MASK>
__device__ __forceinline__ void exp64(const uint32_t (&va)[32], const uint32_t (&vb)[32], int c,
                                      int lo_c, int hi_c, float s_mul, float cap_mul, float m_eff,
                                      float2& rs, uint32_t (&pw)[32]) {
  const float2 mul2 = make_float2(s_mul, s_mul), neg_m = make_float2(-m_eff, -m_eff);
  const unsigned span = hi_c > lo_c ? (unsigned)(hi_c - lo_c) : 0u;
  const float ninf = __int_as_float(0xff800000);
  float2 acc[2] = {rs, make_float2(0.0f, 0.0f)};  // two independent partial sums
#pragma unroll
  for (int g = 0; g < 32; g += 8) {
    float2 x[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int e = 2 * (g + k);
      const float2 sc = make_float2(col_val(va, vb, e), col_val(va, vb, e + 1));
      if (CAP) {
        x[k].x = cap_mul * tanh_via_exp2(sc.x * s_mul) - m_eff;
        x[k].y = cap_mul * tanh_via_exp2(sc.y * s_mul) - m_eff;
      } else {
        x[k] = ffma2(sc, mul2, neg_m);
      }
      if (MASK != kMaskNone) {
        x[k].x = col_visible<MASK>(c + e, lo_c, hi_c, span) ? x[k].x : ninf;
        x[k].y = col_visible<MASK>(c + e + 1, lo_c, hi_c, span) ? x[k].y : ninf;
      }
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) x[k] = make_float2(ex2_approx(x[k].x), ex2_approx(x[k].y));
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      acc[k & 1] = fadd2(acc[k & 1], x[k]);
      pw[g + k] = pack2<T>(x[k].x, x[k].y);
    }
  }
  rs = fadd2(acc[0], acc[1]);
}

}  // namespace pva
