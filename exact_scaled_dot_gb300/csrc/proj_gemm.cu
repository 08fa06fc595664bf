// proj_gemm.cu -- the linear projections on either side of attention, on
// sm_103a tensor cores ("Appendix A.10 -- Attention matrices and
// backpropagation", eqs. A.10.10-A.10.11):
//   forward         Q = X W_Q,  K = X W_K,  V = X W_V            (A.10.10)
//   weight grads    G_W = X^T G  for each projection             (A.10.11)
//   input grad      G_X = G_Q W_Q^T + G_K W_K^T + G_V W_V^T      (A.10.11)
// All are one kernel: C = sum_s A_s B_s over up to three sources, bf16
// operands, fp32 accumulation in tensor memory.  Matrices are row-major in
// memory; an operand is "K-major" when its contraction index is the
// contiguous one and "MN-major" otherwise, and the MMA reads either form
// straight from the swizzled shared-memory tiles TMA writes:
//   Y  = X W      A = X   [T][D]  K-major,   B = W  [D][N]  MN-major
//   dW = X^T G    A = X   [T][D]  MN-major,  B = G  [T][N]  MN-major
//   dX = G W^T    A = G   [T][N]  K-major,   B = W  [D][N]  K-major
//
// CTA: one 128 x 256 output tile, 256 threads.  warp 0 TMA producer (two
// stages of 64 contraction steps: A 16 KB + B 32 KB), warp 1 MMA issuer
// (converged, one elected lane issues; M=128, N=256, four K=16 products per
// stage), warps 4-7 epilogue (thread = output row = TMEM lane).  96 KB of shared memory and 256 tensor
// memory columns, so two CTAs share an SM and one's epilogue overlaps the
// other's products.  Contraction tails, rows and columns past the matrix
// edges read as zeros (TMA bounds fill); the epilogue writes only inside C.
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "f16range.cuh"
#include "ptx.cuh"

namespace esd {
namespace {

constexpr int kGM = 128, kGN = 256, kGK = 64, kGStages = 2;

struct GemmCfg {
  static constexpr int kABytes = kGM * kGK * 2;   // 16 KB
  static constexpr int kBBytes = kGN * kGK * 2;   // 32 KB
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kOffBar = kGStages * kStageBytes;
  static constexpr int kBarFull = 0;                    // [stages]
  static constexpr int kBarEmpty = kBarFull + kGStages; // [stages]
  static constexpr int kBarAcc = kBarEmpty + kGStages;
  static constexpr int kBarDrain = kBarAcc + 1;
  static constexpr int kNumBars = kBarDrain + 1;
  static constexpr int kOffTmemSlot = kOffBar + kNumBars * 8;
  static constexpr int kOffAbort = kOffTmemSlot + 4;
  static constexpr int kSmemBytes = kOffAbort + 4 + 1024;   // slack for 1024-byte alignment
  static constexpr uint32_t kTmemCols = 256;
  static_assert(2 * kSmemBytes <= 232448, "two CTAs per SM");
};

template <bool AMN, bool BMN, bool OUTF32>
__global__ void __launch_bounds__(256, 2)
proj_gemm_kernel(const __grid_constant__ CUtensorMap tA0, const __grid_constant__ CUtensorMap tB0,
                 const __grid_constant__ CUtensorMap tA1, const __grid_constant__ CUtensorMap tB1,
                 const __grid_constant__ CUtensorMap tA2, const __grid_constant__ CUtensorMap tB2,
                 const __grid_constant__ GemmParams p) {
  using C = GemmCfg;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  auto bar = [&](int idx) -> uint32_t { return sbase + C::kOffBar + 8 * idx; };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffAbort);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffTmemSlot);
  const uint32_t warp = warp_id();
  const uint32_t lane = lane_id();
  const int n0 = static_cast<int>(blockIdx.x) * kGN;
  const int64_t m0 = static_cast<int64_t>(blockIdx.y) * kGM;
  int steps[3], total = 0;
  for (int s = 0; s < 3; ++s) {
    steps[s] = s < p.nsrc ? (p.K[s] + kGK - 1) / kGK : 0;
    total += steps[s];
  }

  if (threadIdx.x == 0) {
    for (int s = 0; s < kGStages; ++s) {
      mbar_init(bar(C::kBarFull + s), 1);
      mbar_init(bar(C::kBarEmpty + s), 1);
    }
    mbar_init(bar(C::kBarAcc), 1);
    mbar_init(bar(C::kBarDrain), 1);
    fence_mbar_init();
    *abort_flag = status_blocks(p.status) ? 2 : 0;
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  const uint64_t limit = p.wait_limit_ns;

  if (warp == 0) {
    // ============================ TMA producer ============================
    if (lane == 0 && *abort_flag == 0 && total > 0) {
      int issued[kGStages] = {};
      int it = 0;
      bool ok = true;
      for (int s = 0; s < 3 && ok; ++s) {
        const CUtensorMap* ta = s == 0 ? &tA0 : (s == 1 ? &tA1 : &tA2);
        const CUtensorMap* tb = s == 0 ? &tB0 : (s == 1 ? &tB1 : &tB2);
        if (steps[s] > 0) {
          tma_prefetch_map(ta);
          tma_prefetch_map(tb);
        }
        for (int kt = 0; kt < steps[s]; ++kt, ++it) {
          const int st = it % kGStages;
          ok = mbar_wait(bar(C::kBarEmpty + st), static_cast<uint32_t>(((it / kGStages) & 1) ^ 1), abort_flag,
                         limit);
          if (!ok) break;
          const uint32_t a_dst = sbase + st * C::kStageBytes, b_dst = a_dst + C::kABytes;
          mbar_arrive_expect_tx(bar(C::kBarFull + st), C::kStageBytes);
          const int k0 = kt * kGK;
          if (!AMN) {
            tma_load_2d(a_dst, ta, bar(C::kBarFull + st), k0, static_cast<int32_t>(m0));
          } else {
            for (int h = 0; h < kGM / 64; ++h)
              tma_load_2d(a_dst + h * 8192, ta, bar(C::kBarFull + st), static_cast<int32_t>(m0) + 64 * h, k0);
          }
          if (!BMN) {
            tma_load_2d(b_dst, tb, bar(C::kBarFull + st), k0, n0);
          } else {
            for (int q = 0; q < kGN / 64; ++q)
              tma_load_2d(b_dst + q * 8192, tb, bar(C::kBarFull + st), n0 + 64 * q, k0);
          }
          ++issued[st];
        }
      }
      if (*abort_flag) {
        int no_abort = 0;
        for (int st = 0; st < kGStages; ++st)
          if (issued[st]) mbar_wait(bar(C::kBarFull + st), (issued[st] - 1) & 1, &no_abort, limit);
      }
    }
  } else if (warp == 1) {
    // ============================ MMA issuer =============================
    // The whole warp follows the schedule (waits end in a vote) and one
    // elected lane issues, so that descriptors stay warp-uniform.
    if (__all_sync(0xffffffffu, *abort_flag == 0) && total > 0) {
      constexpr uint32_t kIdesc = idesc_bf16_f32(kGM, kGN, AMN, BMN);
      // K-major tiles step 32 bytes per K=16 product inside the 128-byte
      // swizzle row; MN-major tiles step 16 rows (2048 bytes), their 64-wide
      // blocks 8 KB apart.
      const SmemDesc da0 = AMN ? sw128_desc_words(sbase, 8192, 1024) : sw128_desc_words(sbase, 16, 1024);
      const SmemDesc db0 = BMN ? sw128_desc_words(sbase + C::kABytes, 8192, 1024)
                               : sw128_desc_words(sbase + C::kABytes, 16, 1024);
      constexpr uint32_t kStepA = AMN ? 2048 : 32, kStepB = BMN ? 2048 : 32;
      bool ok = true;
      for (int it = 0; it < total && ok; ++it) {
        const int st = it % kGStages;
        ok = __all_sync(0xffffffffu,
                        mbar_wait(bar(C::kBarFull + st), static_cast<uint32_t>((it / kGStages) & 1), abort_flag, limit));
        if (!ok) break;
        tc_fence_after_sync();
        const SmemDesc da = desc_step(da0, st * C::kStageBytes), db = desc_step(db0, st * C::kStageBytes);
#pragma unroll
        for (int kk = 0; kk < kGK / 16; ++kk)
          umma_ss_we(tmem, desc_step(da, kk * kStepA), desc_step(db, kk * kStepB), kIdesc,
                     (it > 0 || kk > 0) ? 1u : 0u);
        umma_commit_we(bar(C::kBarEmpty + st));
      }
      if (ok) umma_commit_we(bar(C::kBarAcc));
      // Every product issued above must finish before tensor memory is freed.
      int no_abort = 0;
      umma_commit_we(bar(C::kBarDrain));
      mbar_wait(bar(C::kBarDrain), 0, &no_abort, limit);
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ============================== epilogue =============================
    const uint32_t quad = warp & 3;
    const int64_t m = m0 + quad * 32 + lane;
    bool ok = *abort_flag == 0;
    if (ok && total > 0) {
      ok = __all_sync(0xffffffffu, mbar_wait(bar(C::kBarAcc), 0, abort_flag, limit));
      tc_fence_after_sync();
    }
    if (ok) {
      const uint32_t tq = tmem + ((quad * 32u) << 16);
      uint32_t r[32];
#pragma unroll 1
      for (int c = 0; c < kGN / 32; ++c) {
        const int nc = n0 + c * 32;
        if (nc >= p.N) break;   // uniform across the CTA
        if (total > 0) {
          tmem_ld32(tq + c * 32, r);
        } else {
#pragma unroll
          for (int k = 0; k < 32; ++k) r[k] = 0u;
        }
        if (m < p.M) {
          if (OUTF32) {
            float* row = static_cast<float*>(p.C) + m * p.ldc + nc;
#pragma unroll
            for (int v = 0; v < 8; ++v)
              if (nc + 4 * v < p.N)
                *reinterpret_cast<float4*>(row + 4 * v) =
                    make_float4(__uint_as_float(r[4 * v]), __uint_as_float(r[4 * v + 1]),
                                __uint_as_float(r[4 * v + 2]), __uint_as_float(r[4 * v + 3]));
          } else {
            __nv_bfloat16* row = static_cast<__nv_bfloat16*>(p.C) + m * p.ldc + nc;
#pragma unroll
            for (int v = 0; v < 4; ++v)
              if (nc + 8 * v < p.N)
                *reinterpret_cast<uint4*>(row + 8 * v) = make_uint4(
                    pack_bf16x2(__uint_as_float(r[8 * v]), __uint_as_float(r[8 * v + 1])),
                    pack_bf16x2(__uint_as_float(r[8 * v + 2]), __uint_as_float(r[8 * v + 3])),
                    pack_bf16x2(__uint_as_float(r[8 * v + 4]), __uint_as_float(r[8 * v + 5])),
                    pack_bf16x2(__uint_as_float(r[8 * v + 6]), __uint_as_float(r[8 * v + 7])));
          }
        }
      }
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, C::kTmemCols);
  }
  if (threadIdx.x == 0 && *abort_flag == 1) record_status(p.status, ATTN_ERR_TIMEOUT);
}

template <bool AMN, bool BMN, bool OUTF32>
cudaError_t launch_gemm_t(const CUtensorMap* tA, const CUtensorMap* tB, const GemmParams& p, cudaStream_t stream) {
  auto kern = proj_gemm_kernel<AMN, BMN, OUTF32>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, GemmCfg::kSmemBytes);
  if (e != cudaSuccess) return e;
  dim3 grid(static_cast<unsigned>((p.N + kGN - 1) / kGN), static_cast<unsigned>((p.M + kGM - 1) / kGM));
  kern<<<grid, 256, GemmCfg::kSmemBytes, stream>>>(tA[0], tB[0], tA[1], tB[1], tA[2], tB[2], p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_proj_gemm(int kind, const CUtensorMap* tA, const CUtensorMap* tB, const GemmParams& p,
                             cudaStream_t stream) {
  switch (kind) {
    case kGemmXW: return launch_gemm_t<false, true, false>(tA, tB, p, stream);
    case kGemmXtG: return launch_gemm_t<true, true, true>(tA, tB, p, stream);
    case kGemmGWt: return launch_gemm_t<false, false, false>(tA, tB, p, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace esd
