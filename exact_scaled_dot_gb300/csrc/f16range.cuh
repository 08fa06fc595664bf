// f16range.cuh -- power-of-two scaling that keeps bf16 operands exact when
// they are re-encoded as fp16 for the tensor cores.
//
// bf16 has fp32's exponent range and 8 significant bits; fp16 has 11
// significant bits but only the range up to 65504, with normal numbers down
// to 2^-14 and a subnormal grid of 2^-24 below that.  A bf16 value x
// therefore converts to fp16 exactly when 2^-17 <= |x| <= 65504 (down to
// 2^-17 the subnormal grid still holds 8 significant bits); above the range
// it saturates, below it loses bits and finally becomes 0.  Unscaled, legal
// inputs such as gradients of 1e-6 or values of 1e5 would be changed.
//
// So every fp16 operand tile carries an exponent e, x16 = x 2^e, chosen from
// the tile's largest magnitude M so that 2^11 <= M 2^e < 2^15: the largest
// entries land near the top of the fp16 range and every entry down to about
// 2^-28 M is exact.  e is a multiple of 4, so that tiles of similar scale
// (the maxima of unit-variance tiles lie around 4) share one exponent.
// Products of scaled operands are unscaled by exact powers of two.  e is
// clamped to [-kExpLimit, kExpLimit] so that every combination of a few
// exponents stays a normal fp32 power of two; a tile whose M is 2^46 or more
// then saturates, which the kernels report as ATTN_ERR_RANGE.  An all-zero
// tile gets the sentinel kExpZero: it needs no scale, and consumers leave it
// out of the minima they take over tiles.
#pragma once

#include <cmath>
#include <cstdint>

#include "../../include/attn.h"

namespace esd {

constexpr int kExpLimit = 30;
constexpr int kExpZero = 31;

// Exponent of a tile whose largest magnitude is M (M >= 0; an fp32 value, or
// the bits of a bf16 value shifted into an fp32).  Non-finite M (the tile
// holds Inf or NaN) gets 0: such inputs give non-finite results anyway.
__host__ __device__ __forceinline__ int f16_tile_exponent(float M) {
  if (M == 0.f) return kExpZero;
  if (!(M < INFINITY)) return 0;
  int E;
  frexpf(M, &E);   // M = m 2^E, m in [0.5, 1): M < 2^E
  int e = 15 - E;
  e = e >= 0 ? e & ~3 : -((-e + 3) & ~3);   // down to a multiple of 4: 2^11 <= M 2^e < 2^15
  return e < -kExpLimit ? -kExpLimit : (e > kExpLimit ? kExpLimit : e);
}

// True when a tile with largest magnitude M saturates in fp16 at exponent e.
__host__ __device__ __forceinline__ bool f16_saturates(float M, int e) {
  return M < INFINITY && e != kExpZero && ldexpf(M, e) > 65504.f;
}

// The largest magnitude among the eight bf16 values of a 16-byte chunk,
// folded into `m` as two 16-bit lanes of magnitude bits (a non-negative bf16
// orders like its bits).
__device__ __forceinline__ uint32_t bf16_absmax_fold(uint32_t m, uint4 u) {
  m = __vmaxu2(m, u.x & 0x7FFF7FFFu);
  m = __vmaxu2(m, u.y & 0x7FFF7FFFu);
  m = __vmaxu2(m, u.z & 0x7FFF7FFFu);
  return __vmaxu2(m, u.w & 0x7FFF7FFFu);
}

// The folded lanes as one non-negative fp32 value.
__device__ __forceinline__ float bf16_absmax_value(uint32_t m) {
  const uint32_t a = m & 0xFFFFu, b = m >> 16;
  return __uint_as_float((a > b ? a : b) << 16);
}

// Record a device-side condition in the status word.  A wait that timed out
// takes precedence over a range report, since it makes later kernels skip
// their work; a range report only fills an empty word.
__device__ __forceinline__ void record_status(unsigned int* status, unsigned int code) {
  const unsigned int old = atomicCAS(status, 0u, code);
  if (code == static_cast<unsigned int>(ATTN_ERR_TIMEOUT) && old == static_cast<unsigned int>(ATTN_ERR_RANGE))
    atomicCAS(status, old, code);
}

// Kernels skip their work only after a timeout, not after a range report.
__device__ __forceinline__ bool status_blocks(const unsigned int* status) {
  return *reinterpret_cast<const volatile unsigned int*>(status) == static_cast<unsigned int>(ATTN_ERR_TIMEOUT);
}

}  // namespace esd
