// rope.cu -- rotary position embedding of query and key rows, and its
// inverse for their gradients ("Chapter 15 -- matrix formulas", section
// 15.6; "Chapter 31 -- attention backprop", section 5).
//
// Each row x of width d is split into 2-D blocks (x_2k, x_2k+1), k < d/2, and
// block k is rotated by the angle a = pos * w_k, w_k = base^(-2k/d):
//   x'_2k   = x_2k cos a - x_2k+1 sin a
//   x'_2k+1 = x_2k sin a + x_2k+1 cos a          (column-vector rotation R(a)).
// Then R_i^T R_j = R((j - i) w): the rotated dot product depends on the
// position difference only.  The map is orthogonal for a fixed position, so
// the gradient of a rotated row is the upstream gradient rotated back by -a
// (inverse = 1).
//
// Memory-bound: one launch rotates one tensor, or two that share tokens and
// positions (queries and keys).  Every thread takes 8 elements (four blocks)
// of one token, loads those 16 bytes from a group of up to 8 heads of the
// token, computes the four angles once (they depend on the position and the
// block only) and rotates and stores the group.
//
// The angle and the products come from rotary.cuh, shared with the cos/sin
// tables and the rotations fused into the attention kernels.
#include <cstdint>
#include <cuda_runtime.h>

#include "common.cuh"
#include "ptx.cuh"
#include "rotary.cuh"

namespace esd {
namespace {

// One or two token-major tensors that share tokens and positions (the
// queries and keys of a batch), rotated in one launch: the work items of
// tensor 0 come first, then those of tensor 1.
struct RopeParams {
  int64_t tokens;
  int32_t d;             // row width (a multiple of 8)
  int32_t inverse;       // rotate by -a
  int32_t heads[2];      // rows per token of each tensor (0: no second tensor)
  const uint4* x[2];     // bf16 rows, 8 elements per uint4
  uint4* y[2];
  const int32_t* pos;    // [tokens] token positions
  float w_hi[64];        // w_k = base^(-2k/d), k < d/2, rounded to fp32
  float w_lo[64];        // w_k - w_hi[k], rounded to fp32
};

constexpr int kHeadGroup = 8;

__host__ __device__ __forceinline__ int64_t rope_items(int64_t tokens, int heads, int d) {
  return tokens * ((heads + kHeadGroup - 1) / kHeadGroup) * (d / 8);
}

__global__ void __launch_bounds__(256) rope_kernel(const __grid_constant__ RopeParams p) {
  const int per_row = p.d / 8;
  const int64_t items0 = rope_items(p.tokens, p.heads[0], p.d);
  const int64_t total = items0 + rope_items(p.tokens, p.heads[1], p.d);
  for (int64_t u0 = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; u0 < total;
       u0 += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const bool second = u0 >= items0;
    const int64_t u = second ? u0 - items0 : u0;
    const int heads = second ? p.heads[1] : p.heads[0];
    const uint4* x = second ? p.x[1] : p.x[0];   // y may equal x (in place)
    uint4* y = second ? p.y[1] : p.y[0];
    const int groups = (heads + kHeadGroup - 1) / kHeadGroup;
    const int64_t tg = u / per_row;                      // (token, head group)
    const int c = static_cast<int>(u - tg * per_row);    // 8-element chunk: blocks 4c .. 4c+3
    const int64_t tok = tg / groups;
    const int h0 = static_cast<int>(tg - tok * groups) * kHeadGroup;
    const int h1 = h0 + kHeadGroup < heads ? h0 + kHeadGroup : heads;
    // Every row of the group is requested before the angles are formed, so
    // a thread keeps up to 8 x 16 bytes in flight.
    const int64_t base = tok * heads * per_row + c;
    const int32_t pos = p.pos[tok];
    uint4 v[kHeadGroup];
#pragma unroll
    for (int j = 0; j < kHeadGroup; ++j)
      if (h0 + j < h1) v[j] = x[base + static_cast<int64_t>(h0 + j) * per_row];
    float wh[4], wl[4];
    rope_freqs4(p.w_hi, p.w_lo, c, wh, wl);
    float4 t0, t1;
    rope_angles4(pos, wh, wl, t0, t1);
    if (p.inverse) rope_transpose(t0, t1);
#pragma unroll
    for (int j = 0; j < kHeadGroup; ++j) {
      if (h0 + j >= h1) break;
      y[base + static_cast<int64_t>(h0 + j) * per_row] = rot_bf16x8(v[j], t0, t1);
    }
  }
}

__global__ void __launch_bounds__(256) rope_prep_kernel(const __grid_constant__ RopePrepParams p) {
  rope_prep_range(p, static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x,
                  static_cast<int64_t>(gridDim.x) * blockDim.x);
}

}  // namespace

cudaError_t launch_rope_prep(const RopePrepParams& p, cudaStream_t stream) {
  int64_t blocks = ((p.seg[0].tokens + p.seg[1].tokens) * (p.d / 8) + 255) / 256;
  if (blocks > 152 * 64) blocks = 152 * 64;
  if (blocks < 1) blocks = 1;
  rope_prep_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_rope(int64_t tokens, int d, int heads_a, int heads_b, const int32_t* pos, const float* w_hi,
                        const float* w_lo, int inverse, const void* xa, void* ya, const void* xb, void* yb, cudaStream_t stream) {
  RopeParams p{};
  p.tokens = tokens;
  p.d = d;
  p.inverse = inverse;
  p.heads[0] = heads_a;
  p.heads[1] = heads_b;
  p.x[0] = static_cast<const uint4*>(xa);
  p.y[0] = static_cast<uint4*>(ya);
  p.x[1] = static_cast<const uint4*>(xb);
  p.y[1] = static_cast<uint4*>(yb);
  p.pos = pos;
  for (int k = 0; k < d / 2; ++k) {
    p.w_hi[k] = w_hi[k];
    p.w_lo[k] = w_lo[k];
  }
  int64_t blocks = (rope_items(tokens, heads_a, d) + rope_items(tokens, heads_b, d) + 255) / 256;
  if (blocks > 152 * 64) blocks = 152 * 64;
  if (blocks < 1) blocks = 1;
  rope_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace esd
