// bwd_scale.cuh -- the power-of-two scales of the backward main kernels'
// fp16 operands, shared by the grid kernel (attn_bwd.cu) and the persistent
// kernel (attn_bwd_persist.cu).  What they make exact is set out below; the
// bound on |dS| is that of "Appendix A.10 -- Attention matrices and
// backpropagation", eq. A.10.7 (dS_ij = A_ij (dA_ij - c_i), with |A_ij| <= 1
// and |dA_ij| = |dO_i . v_j| <= ||dO_i|| ||v_j||).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "f16range.cuh"

namespace esd {
namespace {

// The fp16 operand exponents of one key tile's backward work (f16range.cuh):
// K16 = K 2^k and V16 = V 2^v for the key tile, and Q16 = Q 2^q, dO16 = dO 2^o for every
// query tile of its (batch, KV head) group (attn_bwd_group_exp_kernel gives
// all of a group's tiles one q and one o, so no step needs a scale of its
// own).  The products then carry
//   S^T = K16 Q16^T = 2^(k + q) S_raw^T,   dP^T = V16 dO16^T = 2^(v + o) dP^T,
//   dV_acc = P^T dO16 = 2^o dV,
// and dS enters dQ and dK as fp16 dS' = 2^g dS, with g chosen from the bound
// |dS_ij| <= max ||dO_i|| max ||v_j|| + max |D_i| (the preprocess's tile
// maxima and the V tile's row norms) so that |dS'| < 2^14: no fp16
// overflow, and small gradients stay far from the fp16 subnormals.  Then
//   dQ_acc = dS' K16 = 2^(g + k) dS K,   dK_acc = dS'^T Q16 = 2^(g + q) dS^T Q,
// all unscaled exactly.  Every exponent lies in [-30, 30], so each derived
// multiplier is a normal fp32 power of two.
struct CtaScale {
  float mv;        // max_j ||v_j|| over the key tile
  int v, q, o, g;
  bool overflow;   // the bound needed g < -30: dS' may saturate
};

// From the key tile's maxima (max ||v_j||, and max ||dO_i||, max |D_i| over
// the query tiles its steps visit) and the group's exponents (q, o).
__device__ __forceinline__ CtaScale cta_scale_of(float mv, float mdo, float md, float2 qo) {
  CtaScale c;
  c.mv = mv;
  c.v = f16_tile_exponent(c.mv);
  if (c.v == kExpZero) c.v = 0;
  c.q = static_cast<int>(qo.x);
  c.o = static_cast<int>(qo.y);
  int g = kExpLimit;
  const float bound = mdo * c.mv + md;
  if (bound > 0.f && bound < INFINITY) {
    int E;
    frexpf(bound, &E);   // bound < 2^E, so |dS| 2^(14 - E) < 2^14
    g = min(g, 14 - E);
  }
  c.overflow = g < -kExpLimit;
  c.g = c.overflow ? -kExpLimit : g;
  return c;
}

}  // namespace
}  // namespace esd
