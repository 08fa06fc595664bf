// rotary.cuh -- the arithmetic of the rotary position embedding, shared by
// every kernel that rotates ("Chapter 15 -- matrix formulas", section 15.6;
// "Chapter 31 -- attention backprop", section 5).
//
// Block k of a row (its components 2k, 2k+1) turns by the angle
// a = pos * w_k, w_k = base^(-2k/d), with the column-vector rotation
//   y_2k   = x_2k cos a - x_2k+1 sin a
//   y_2k+1 = x_2k sin a + x_2k+1 cos a,
// and a gradient turns back by -a (the transpose).  The separate rotation
// pass, the cos/sin tables and the rotations fused into the attention
// kernels all form the angle with reduced_angle, its cosine and sine with
// rope_cos_sin and the products with rot_block, so a row rotated in any of
// them has the same bits.
#pragma once

#include <cstdint>

#include "common.cuh"
#include "ptx.cuh"

namespace esd {

constexpr int kRopeHeadGroup = 8;   // rows rotated per work item with one set of angles

// 2 pi = C1 + C2 + C3: C1 with trailing zero bits (8 significant bits), C2
// the fp32 rounding of the rest, C3 that rounding's residual.
constexpr float kTwoPiC1 = 6.28125f;
constexpr float kTwoPiC2 = static_cast<float>(6.283185307179586476925 - 6.28125);
constexpr float kTwoPiC3 = static_cast<float>(6.283185307179586476925 - 6.28125 - static_cast<double>(kTwoPiC2));
constexpr float kInvTwoPi = 0.15915494309189535f;

// p (w_hi + w_lo) reduced modulo 2 pi, to about single precision of the
// reduced angle for every |p| < 2^24.  w arrives as w_hi + w_lo (w_lo the
// rounding residual of w_hi, both from the double-precision frequency), the
// product p w_hi is split exactly into hi + lo with an fma, lo collects
// p w_lo, and hi is reduced by a three-constant Cody-Waite scheme.  For
// |hi| < 2^24 the quotient k is below 2^22 and fmaf(-k, C1, hi) is exact (the
// difference is at most a few thousand and lies on the grid of the finer of
// hi's unit in the last place and C1's 2^-5); the C2 and C3 steps and the
// final additions round a few times near |r| <= pi.
__device__ __forceinline__ float reduced_angle(int32_t pos, float w_hi, float w_lo) {
  const float p = static_cast<float>(pos);      // exact for |pos| < 2^24
  const float hi = p * w_hi;
  const float lo = fmaf(p, w_lo, fmaf(p, w_hi, -hi));   // p w_hi = hi + its residual, plus p w_lo
  const float k = rintf(hi * kInvTwoPi);
  float r = fmaf(-k, kTwoPiC1, hi);
  r = fmaf(-k, kTwoPiC2, r);
  r = fmaf(-k, kTwoPiC3, r);
  return r + lo;
}

// Cosine and sine of a reduced angle (|r| <= pi and a little): the
// hardware's sine and cosine, whose absolute error on [-pi, pi] is about
// 4e-7, comparable to the reduction's own few 1e-7 and far below the 2^-9
// relative rounding of the bf16 results.
__device__ __forceinline__ void rope_cos_sin(float r, float& c, float& s) { __sincosf(r, &s, &c); }

// The table entries (cos, sin, cos, sin) of blocks 4c, 4c+1 (t0) and
// 4c+2, 4c+3 (t1) at position pos, from the four blocks' frequencies.
__device__ __forceinline__ void rope_angles4(int32_t pos, const float (&w_hi)[4], const float (&w_lo)[4], float4& t0,
                                             float4& t1) {
  float c[4], s[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) rope_cos_sin(reduced_angle(pos, w_hi[q], w_lo[q]), c[q], s[q]);
  t0 = make_float4(c[0], s[0], c[1], s[1]);
  t1 = make_float4(c[2], s[2], c[3], s[3]);
}

// One block (x0, x1) turned by the angle whose cosine is c and sine s.  The
// products are rounded one by one (no contraction the compiler may choose
// differently in different kernels).  The transpose is rot_block(x0, x1, c, -s).
__device__ __forceinline__ void rot_block(float x0, float x1, float c, float s, float& y0, float& y1) {
  y0 = __fmaf_rn(x0, c, -__fmul_rn(x1, s));
  y1 = __fmaf_rn(x0, s, __fmul_rn(x1, c));
}

// One packed bf16 block turned and rounded back to bf16.  The same products
// and roundings as rot_block, as two paired instructions: m = x1 (-s, c),
// then y = x0 (c, s) + m.
__device__ __forceinline__ uint32_t rot_bf16x2(uint32_t w, float c, float s) {
  const float x0 = bf16_lo(w), x1 = bf16_hi(w);
  float m0, m1, y0, y1;
  fmul2(m0, m1, x1, x1, -s, c);
  ffma2(y0, y1, x0, x0, c, s, m0, m1);
  return pack_bf16x2(y0, y1);
}

// Eight bf16 values (blocks 4c .. 4c+3 of a row) turned by the table entries
// t0 = (cos, sin, cos, sin) of blocks 4c, 4c+1 and t1 of blocks 4c+2, 4c+3.
__device__ __forceinline__ uint4 rot_bf16x8(uint4 v, float4 t0, float4 t1) {
  return make_uint4(rot_bf16x2(v.x, t0.x, t0.y), rot_bf16x2(v.y, t0.z, t0.w), rot_bf16x2(v.z, t1.x, t1.y),
                    rot_bf16x2(v.w, t1.z, t1.w));
}

// The four frequencies of blocks 4c .. 4c+3.
__device__ __forceinline__ void rope_freqs4(const float* w_hi, const float* w_lo, int c, float (&wh)[4],
                                            float (&wl)[4]) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    wh[q] = w_hi[4 * c + q];
    wl[q] = w_lo[4 * c + q];
  }
}

// The cosines and sines of the transpose (the turn back): sines negated.
__device__ __forceinline__ void rope_transpose(float4& t0, float4& t1) {
  t0.y = -t0.y;
  t0.w = -t0.w;
  t1.y = -t1.y;
  t1.w = -t1.w;
}

// Rotated copies ahead of the attention kernels (RopePrepParams): work items
// first, first + stride, ...  Item u is an 8-element chunk c (blocks
// 4c .. 4c+3) of one token, the tokens of segment 0 first, then those of
// segment 1.  Each item forms its four angles once and rotates chunk c of
// every head of its token into Y (up to kRopeHeadGroup rows in flight).
__device__ __forceinline__ void rope_prep_range(const RopePrepParams& p, int64_t first, int64_t stride) {
  const int per_row = p.d / 8;
  const int64_t items0 = p.seg[0].tokens * per_row;
  const int64_t total = items0 + p.seg[1].tokens * per_row;
  for (int64_t u0 = first; u0 < total; u0 += stride) {
    const bool second = u0 >= items0;
    const RopeSegment& g = p.seg[second ? 1 : 0];
    const int64_t u = second ? u0 - items0 : u0;
    const int64_t tok = u / per_row;
    const int c = static_cast<int>(u - tok * per_row);
    const int32_t pos = g.pos[tok];
    const uint4* X = static_cast<const uint4*>(g.X);
    uint4* Y = static_cast<uint4*>(g.Y);
    // Element offsets of this token's row of head h: in the caller's tensor
    // (strided) and in the contiguous rotated copy.
    int64_t src0, dst0, dst_h;
    if (p.packed) {
      src0 = tok * g.sx.row;
      dst0 = tok * g.H * p.d;
      dst_h = p.d;
    } else {
      const int64_t b = tok / g.n, i = tok - b * g.n;
      src0 = b * g.H * g.sx.head + i * g.sx.row;
      dst0 = (b * g.H * g.n + i) * p.d;
      dst_h = static_cast<int64_t>(g.n) * p.d;
    }
    uint4 v[kRopeHeadGroup];
#pragma unroll
    for (int h = 0; h < kRopeHeadGroup; ++h)
      if (h < g.H) v[h] = X[(src0 + h * g.sx.head) / 8 + c];
    float wh[4], wl[4];
    rope_freqs4(p.w_hi, p.w_lo, c, wh, wl);
    float4 t0, t1;
    rope_angles4(pos, wh, wl, t0, t1);
    for (int h0 = 0; h0 < g.H; h0 += kRopeHeadGroup) {
      if (h0 > 0) {
#pragma unroll
        for (int h = 0; h < kRopeHeadGroup; ++h)
          if (h0 + h < g.H) v[h] = X[(src0 + (h0 + h) * g.sx.head) / 8 + c];
      }
#pragma unroll
      for (int h = 0; h < kRopeHeadGroup; ++h)
        if (h0 + h < g.H) Y[(dst0 + (h0 + h) * dst_h) / 8 + c] = rot_bf16x8(v[h], t0, t1);
    }
  }
}

}  // namespace esd
