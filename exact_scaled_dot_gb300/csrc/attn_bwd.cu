// attn_bwd.cu -- backward kernels of masked scaled dot-product attention on
// sm_103a.
//
// What they compute ("Appendix A.10 -- Attention matrices and
// backpropagation", eqs. A.10.5-A.10.9; "Chapter 31 -- attention backprop",
// sections 2-4):
//   dV = A^T dO,  dA = dO V^T,  dS = A .* (dA - c) with c_i = rowsum(dO .* O),
//   dQ = scale dS K,  dK = scale dS^T Q,
// with dK and dV summed over the query heads that share a KV head (A.10.5).
// The weights A are never stored: the main kernel rebuilds them from the
// scores and the forward's log-sum-exp, A_ij = exp(scale q_i.k_j - LSE_i)
// (the recomputation the appendix names in section A.10.6).
//
// Four kernels:
//   preprocess  D_i = sum_l dO_il O_il (equal to c_i of A.10.7 because
//               O_i = sum_j A_ij v_j), zeroes the fp32 dQ accumulator and
//               writes Q and dO re-encoded as fp16 (the main kernel's
//               operands), each query tile scaled by a power of two from its
//               largest magnitude (f16range.cuh).
//               O is taken as the bf16 output plus the forward's bf16
//               rounding residual, so D is not limited by the bf16 rounding
//               of O.  Per 128-row query tile it also records max ||dO_i||
//               and max |D_i|, which bound |dS| (below).
//   group exp   brings the fp16 query tiles of each (batch, KV head) group to
//               one exponent for Q and one for dO (usually they agree and
//               nothing is rewritten), so the main kernel's steps share one
//               scale.
//   main        one CTA per (batch, KV head, 128-key tile).  It loops over
//               the query heads of its group and the query tiles that can
//               see its keys, keeps dK and dV in tensor memory for the whole
//               loop, and adds each tile's dS K product into the fp32 dQ
//               accumulator with TMA reduce-add.  (attn_bwd_persist.cu
//               holds the same kernel under a persistent schedule, which the
//               host takes when the items have few steps.)
//   finalize    dQ = scale * accumulator, rounded to bf16.
//
// Main-kernel warp roles (512 threads):
//   warp 0      TMA producer: the K and V tile once, then the fp16 Q tile
//               of every step into a two-stage ring and its fp16 dO tile
//               into a single stage (dO(s) is dead once dV(s) is done).
//   warps 1, 3  MMA issuers (one elected lane issues).
//   warps 4-11  two "score" warpgroups, one per 64-query half of the step,
//               thread = key row = TMEM lane:
//               P^T = exp2(S^T scale log2e - LSE log2e) and
//               dS = P (dP - D), P^T written back to tensor memory (for
//               dV) and dS to shared memory (for dQ and dK).
//   warps 12-15 convert K and V to fp16 in shared memory (each scaled by a
//               power of two of its own), read dQ out of tensor memory into
//               the accumulator and write the final dK, dV.
// The producer/MMA and read-out warpgroups hand registers to the score
// warpgroups (setmaxnreg), which hold 64 scores and the fp16 weights of a
// step at once.
//
// Precision of the dS products.  dQ_i = scale sum_j dS_ij k_j sums terms
// that largely cancel when a softmax row is sharply peaked, so rounding dS
// to bf16 (8 significant bits) alone can use up most of a 1e-2 error
// budget.  dS therefore enters the dK and dQ products as fp16 (11 bits),
// multiplied by a per-CTA power of two 2^g chosen from the bound
//   |dS_ij| <= P_ij |dP_ij - D_i| <= max_i ||dO_i|| max_j ||v_j|| + max_i |D_i|
// so that |2^g dS| <= 2^14: no fp16 overflow, and small gradients stay far
// from the fp16 subnormal range.  The scale is exact and undone exactly when
// dQ is read out and when dK is written.  Every product runs in fp16 (the
// MMA takes one type for both operands): Q and dO arrive re-encoded by the
// preprocess, K and V are converted once per CTA, each operand multiplied by
// a power of two that brings its largest magnitude to the top of the fp16
// range (CtaScale), so the re-encoding is exact at any input scale; the
// weights P -- one fp16 rounding, used both in dS and as P^T in
// dV = P^T dO -- keep 11 significant bits, where bf16 weights left dV
// errors near the tolerance for keys whose gradient sums a few hundred
// comparable terms.
// Per step (query tile of 128 rows) the products are
//   S^T = K Q^T -> X, dP^T = V dO^T -> Y, dV += P^T dO, dQ = dS K -> Y,
//   dK += dS^T Q,
// where tensor memory holds X [0,128), Y [128,256), dK [256, 256+DH) and
// dV [256+DH, 256+DH+DV).  P^T (fp16) overwrites the first 64 columns of X
// once the scores are consumed; dS goes to shared memory only, where it
// serves both dQ and dK.  dQ reuses Y once the score warps have read dP^T
// out of it, and is read out while dK runs, which leaves X free for the
// next step's scores.
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "f16range.cuh"
#include "ptx.cuh"
#include "rotary.cuh"
#include "bwd_scale.cuh"

namespace esd {
namespace {

template <int DH, int DV>
struct BwdCfg {
  static constexpr int kStages = 2;
  static constexpr int kKTileBytes = kTileN * DH * 2;
  static constexpr int kVTileBytes = kTileN * DV * 2;
  static constexpr int kQTileBytes = kTileM * DH * 2;
  static constexpr int kDOTileBytes = kTileM * DV * 2;
  static constexpr int kDSTileBytes = kTileN * kTileM * 2;
  static constexpr int kBlockBytes = 128 * 128;
  static constexpr int kOffK = 0;
  static constexpr int kOffV = kOffK + kKTileBytes;
  static constexpr int kOffQ = kOffV + kVTileBytes;
  static constexpr int kOffDO = kOffQ + kStages * kQTileBytes;   // one stage: dO(s) is dead after dV(s)
  static constexpr int kOffDS = kOffDO + kDOTileBytes;
  static constexpr int kOffStage = kOffDS + kDSTileBytes;          // dQ staging, 4 warps x 8 KB
  static constexpr int kOffLse = kOffStage + 4 * 2 * 32 * 32 * 4;
  static constexpr int kOffDd = kOffLse + kTileM * 4;
  // Reductions: the score warps' per-warp maxima and exponent extremes
  // (4 warps x 8 floats), the read-out warps' K-tile maxima (4) and the K
  // tile's exponent.
  static constexpr int kOffRed = kOffDd + kTileM * 4;
  static constexpr int kRedK = 32, kRedKExp = 36;
  static constexpr int kOffBar = kOffRed + 256;
  static constexpr int kBarKV = 0;
  static constexpr int kBarQFull = 1;                 // [2]
  static constexpr int kBarQEmpty = kBarQFull + 2;    // [2]
  static constexpr int kBarDOFull = kBarQEmpty + 2;
  static constexpr int kBarDOEmpty = kBarDOFull + 1;
  static constexpr int kBarK16 = kBarDOEmpty + 1;     // K tile re-encoded as fp16
  static constexpr int kBarV16 = kBarK16 + 1;         // V tile re-encoded as fp16 (after the bound read it)
  static constexpr int kBarScale = kBarV16 + 1;       // dS scale bound reduced
  static constexpr int kBarSFull = kBarScale + 1;
  static constexpr int kBarDPFull = kBarSFull + 1;
  static constexpr int kBarPReady = kBarDPFull + 1;
  static constexpr int kBarDSReady = kBarPReady + 1;
  static constexpr int kBarDQFull = kBarDSReady + 1;
  static constexpr int kBarDQFree = kBarDQFull + 1;
  static constexpr int kBarDKDone = kBarDQFree + 1;   // dK(s) done: dS tile free again
  static constexpr int kBarDKDV = kBarDKDone + 1;
  static constexpr int kBarDrain = kBarDKDV + 1;
  static constexpr int kNumBars = kBarDrain + 1;
  static constexpr int kOffTmemSlot = kOffBar + kNumBars * 8;
  static constexpr int kOffAbort = kOffTmemSlot + 4;
  static constexpr int kSmemUsed = kOffAbort + 4;
  static constexpr int kSmemBytes = kSmemUsed + 1024;
  static constexpr int kThreads = 512;
  // Registers per thread: 128 at launch (65536 / 512); the producer/MMA
  // warpgroup gives most of its share to the score and read-out warpgroups
  // (128 x 56 + 256 x 176 + 128 x 96 = 64512 <= 512 x 128).
  static constexpr uint32_t kRegsLaunch = 128;   // 65536 / 512
  static constexpr uint32_t kRegsLow = 64, kRegsScore = 176, kRegsAux = 96;
  static_assert(128 * kRegsLow + 256 * kRegsScore + 128 * kRegsAux <= 512 * kRegsLaunch, "register split");
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kTX = 0, kTY = 128, kTdK = 256, kTdV = 256 + DH;
  // dQ read-out: each read-out warp stages its 32 query rows as boxes of 32
  // rows x 32 fp32 (4 KB) in its own 8 KB of a dedicated staging buffer,
  // two boxes per round, DH / 64 rounds per step.
  static constexpr int kDQBoxCols = 32;
  static constexpr int kDQBoxBytes = 32 * kDQBoxCols * 4;
  static constexpr int kDQBoxes = DH / kDQBoxCols;
  static constexpr int kDQBoxesPerRound = 2;
  static constexpr int kDQRounds = kDQBoxes / kDQBoxesPerRound;
  static constexpr int kDQWarpStage = kDQBoxesPerRound * kDQBoxBytes;
  static_assert(kSmemBytes <= 232448, "shared memory budget");
  static_assert(256 + DH + DV <= 512, "tensor memory budget");
};

// From the score warps' reduction (per warp w: red[4w .. 4w+2] = max
// ||v_j||, max ||dO_i||, max |D_i|) and the group's exponents (q, o).  (One
// out-of-line copy for the two warpgroups that call it.)
__device__ __noinline__ CtaScale cta_scale(const float* red, float2 qo) {
  float mv = 0.f, mdo = 0.f, md = 0.f;
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    mv = fmaxf(mv, red[4 * w]);
    mdo = fmaxf(mdo, red[4 * w + 1]);
    md = fmaxf(md, red[4 * w + 2]);
  }
  return cta_scale_of(mv, mdo, md, qo);
}

template <int DH, int DV, bool PACKED, bool ROPE, bool SPLIT>
__global__ void __launch_bounds__(512, 1)
attn_bwd_main_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                     const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                     const __grid_constant__ CUtensorMap tmdQ, const __grid_constant__ BwdParams p) {
  using C = BwdCfg<DH, DV>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  auto bar = [&](int idx) -> uint32_t { return sbase + C::kOffBar + 8 * idx; };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffAbort);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffTmemSlot);
  float* lse_s = reinterpret_cast<float*>(smem + C::kOffLse);
  float* dd_s = reinterpret_cast<float*>(smem + C::kOffDd);
  float* red_s = reinterpret_cast<float*>(smem + C::kOffRed);

  const uint32_t warp = warp_id();
  const uint32_t lane = lane_id();

  // ---- work item: key tile blockIdx.y of (batch, KV head) blockIdx.x.  The
  // (batch, KV head) index runs fastest, so the first CTAs dispatched are the
  // low key tiles, which under a causal mask see the most query tiles. ----
  const int bkv = blockIdx.x;
  const int b = bkv / p.sh.Hkv;
  const int hkv = bkv - b * p.sh.Hkv;
  const int64_t j0 = static_cast<int64_t>(blockIdx.y) * kTileN;
  const int64_t klen = key_len(p.mask, p.sh.n_k, b);
  const int64_t nq_b = query_len(p.mask, p.sh.n_q, b);
  const int64_t i_first = first_row_seeing_key(p.mask, p.sh.n_q, p.sh.n_k, b, j0);
  const int nqt = static_cast<int>((nq_b + kTileM - 1) / kTileM);
  const int qt_first = static_cast<int>(i_first / kTileM);
  const int per_head = (i_first < nq_b) ? (nqt - qt_first) : 0;
  // dK/dV rows this CTA writes: up to n_k in the padded layout (rows past
  // kv_len get zeros); in the packed layout rows past the sequence belong to
  // another one.
  const int64_t k_row_end = PACKED ? klen : p.sh.n_k;
  // Query-head split (SPLIT): this CTA takes heads [z hps, (z + 1) hps) of
  // the group, z = blockIdx.z.
  const int hps = SPLIT ? p.sh.group / p.hsplit : p.sh.group;
  const int total = per_head * hps;
  const int head0 = hkv * p.sh.group + (SPLIT ? static_cast<int>(blockIdx.z) * hps : 0);
  auto step_head = [&](int s) { return head0 + s / per_head; };
  auto step_q0 = [&](int s) { return (qt_first + s % per_head) * kTileM; };

  if (threadIdx.x == 0) {
    mbar_init(bar(C::kBarKV), 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(C::kBarQFull + s), 1);
      mbar_init(bar(C::kBarQEmpty + s), 1);
    }
    mbar_init(bar(C::kBarDOFull), 1);
    mbar_init(bar(C::kBarDOEmpty), 1);
    mbar_init(bar(C::kBarK16), 128);
    mbar_init(bar(C::kBarV16), 128);
    mbar_init(bar(C::kBarScale), 128);
    mbar_init(bar(C::kBarSFull), 1);
    mbar_init(bar(C::kBarDPFull), 1);
    mbar_init(bar(C::kBarPReady), 256);
    mbar_init(bar(C::kBarDSReady), 256);
    mbar_init(bar(C::kBarDQFull), 1);
    mbar_init(bar(C::kBarDQFree), 128);
    mbar_init(bar(C::kBarDKDone), 1);
    mbar_init(bar(C::kBarDKDV), 2);    // one commit from each MMA issuer
    mbar_init(bar(C::kBarDrain), 2);
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
  auto wait_all = [&](int idx, uint32_t parity) -> bool {
    const bool w = mbar_wait(bar(idx), parity, abort_flag, limit);
    return __all_sync(0xffffffffu, w);
  };
  // The group's exponents (q, o) (attn_bwd_group_exp_kernel).
  auto group_exps = [&]() -> float2 { return p.grpexp[bkv]; };

  if (warp < 4) setmaxnreg_to<C::kRegsLow, C::kRegsLaunch>();
  if (warp == 0) {
    // =========================== TMA producer ===========================
    if (lane == 0 && *abort_flag == 0 && total > 0) {
      tma_prefetch_map(&tmQ);
      tma_prefetch_map(&tmK);
      tma_prefetch_map(&tmV);
      tma_prefetch_map(&tmdO);
      for (int s = 0; s < 2 && s < total; ++s) {
        const TmaYZ yz = q_tma(PACKED, p.lay, p.sh.Hq, b, step_head(s), step_q0(s));
        for (int c = 0; c < DH / 64; ++c) tma_prefetch_l2_3d(&tmQ, c * 64, yz.y, yz.z);
        for (int c = 0; c < DV / 64; ++c) tma_prefetch_l2_3d(&tmdO, c * 64, yz.y, yz.z);
      }
      const TmaYZ kyz = k_tma(PACKED, p.lay, p.sh.Hkv, b, hkv, static_cast<int>(j0));
      mbar_arrive_expect_tx(bar(C::kBarKV), C::kKTileBytes + C::kVTileBytes);
      for (int c = 0; c < DH / 64; ++c)
        tma_load_3d(sbase + C::kOffK + c * C::kBlockBytes, &tmK, bar(C::kBarKV), c * 64,
                    kyz.y, kyz.z);
      for (int c = 0; c < DV / 64; ++c)
        tma_load_3d(sbase + C::kOffV + c * C::kBlockBytes, &tmV, bar(C::kBarKV), c * 64,
                    kyz.y, kyz.z);
      int q_issued[2] = {0, 0}, do_issued = 0;
      for (int s = 0; s < total; ++s) {
        const int st = s & 1;
        const uint32_t ph = static_cast<uint32_t>(((s >> 1) & 1) ^ 1);
        const TmaYZ yz = q_tma(PACKED, p.lay, p.sh.Hq, b, step_head(s), step_q0(s));
        if (!mbar_wait(bar(C::kBarQEmpty + st), ph, abort_flag, limit)) break;
        mbar_arrive_expect_tx(bar(C::kBarQFull + st), C::kQTileBytes);
        for (int c = 0; c < DH / 64; ++c)
          tma_load_3d(sbase + C::kOffQ + st * C::kQTileBytes + c * C::kBlockBytes, &tmQ,
                      bar(C::kBarQFull + st), c * 64, yz.y, yz.z);
        ++q_issued[st];
        // One dO stage: dO(s) is read by dP(s) and dV(s) only, so the next
        // tile loads as soon as dV(s) is done, well before dP(s+1).
        if (s > 0 && !mbar_wait(bar(C::kBarDOEmpty), static_cast<uint32_t>((s - 1) & 1), abort_flag, limit)) break;
        mbar_arrive_expect_tx(bar(C::kBarDOFull), C::kDOTileBytes);
        for (int c = 0; c < DV / 64; ++c)
          tma_load_3d(sbase + C::kOffDO + c * C::kBlockBytes, &tmdO, bar(C::kBarDOFull), c * 64, yz.y, yz.z);
        ++do_issued;
        // Warm L2 with the tiles of step s + 2: their shared-memory stage is
        // only free once step s has finished, which leaves too little time to
        // hide a load from HBM.
        if (s + 2 < total) {
          const TmaYZ yz2 = q_tma(PACKED, p.lay, p.sh.Hq, b, step_head(s + 2), step_q0(s + 2));
          for (int c = 0; c < DH / 64; ++c) tma_prefetch_l2_3d(&tmQ, c * 64, yz2.y, yz2.z);
          for (int c = 0; c < DV / 64; ++c) tma_prefetch_l2_3d(&tmdO, c * 64, yz2.y, yz2.z);
        }
      }
      if (*abort_flag) {
        int no_abort = 0;
        mbar_wait(bar(C::kBarKV), 0, &no_abort, limit);
        for (int st = 0; st < 2; ++st) {
          if (q_issued[st]) mbar_wait(bar(C::kBarQFull + st), (q_issued[st] - 1) & 1, &no_abort, limit);
        }
        if (do_issued) mbar_wait(bar(C::kBarDOFull), (do_issued - 1) & 1, &no_abort, limit);
      }
    }
  } else if (warp == 1 || warp == 3) {
    // =========================== MMA issuers ============================
    // Two issuers on two SM sub-partitions split each step's products:
    //   warp 1 (A):  dV(s) | S(s+1) -> X | dP(s+1) -> Y
    //   warp 3 (B):  dQ(s) -> Y, dK(s)
    // An MMA issue takes several instructions of the issuing thread, and the
    // score and read-out warps sharing a sub-partition leave it only part of
    // the issue slots; two issuers halve the instructions each one needs.
    // Ordering across the two:
    //   X: dV(s) reads P^T(s) before S(s+1) overwrites it (both A, in order).
    //   Y: dP(s) [A] -> score warps read it -> dQ(s) [B, after dS ready]
    //      -> read-out -> dP(s+1) [A, after dQ free].
    //   dS tile: dQ(s), dK(s) [B] read it; the score warps rewrite it only
    //      after dP(s+1) has landed, and A issues dP(s+1) after B's dK(s)
    //      has completed.
    //   Q(s) stage: S(s) [A] completed before the scores of step s were
    //      seen, so B's commit after dK(s) releases it.
    // Each issuer warp runs converged: all lanes wait (with a vote) and one
    // elected lane issues, so that descriptors and tensor-memory addresses
    // stay warp-uniform and the issue keeps its rate under the score warps'
    // pressure.
    const bool issuer_a = warp == 1;
    if (__all_sync(0xffffffffu, *abort_flag == 0) && total > 0) {
      constexpr uint32_t kIdS = idesc_f16_f32(128, 128, false, false);    // S^T = K Q^T (fp16)
      constexpr uint32_t kIdDP = idesc_f16_f32(128, 128, false, false);   // dP^T = V dO^T (fp16)
      constexpr uint32_t kIdDV = idesc_f16_f32(128, DV, false, true);     // dV += P^T dO (fp16)
      constexpr uint32_t kIdDK = idesc_f16_f32(128, DH, false, true);     // dK += dS^T Q
      constexpr uint32_t kIdDQ = idesc_f16_f32(128, DH, true, true);      // dQ = dS K
      bool ok = wait_all(C::kBarK16, 0);
      // Shared-memory descriptors as base words plus steps (K-major operands:
      // leading offset 16; MN-major: the next 64-column block), so that few
      // instructions sit between two MMAs; the loops stay rolled so that the
      // kernel's code fits the instruction cache next to the other warps.
      const SmemDesc dK_k = sw128_desc_words(sbase + C::kOffK, 16, 1024);
      const SmemDesc dK_mn = sw128_desc_words(sbase + C::kOffK, C::kBlockBytes, 1024);
      const SmemDesc dV_k = sw128_desc_words(sbase + C::kOffV, 16, 1024);
      const SmemDesc dQ_k = sw128_desc_words(sbase + C::kOffQ, 16, 1024);
      const SmemDesc dQ_mn = sw128_desc_words(sbase + C::kOffQ, C::kBlockBytes, 1024);
      const SmemDesc dDO_k = sw128_desc_words(sbase + C::kOffDO, 16, 1024);
      const SmemDesc dDO_mn = sw128_desc_words(sbase + C::kOffDO, C::kBlockBytes, 1024);
      const SmemDesc dDS_k = sw128_desc_words(sbase + C::kOffDS, 16, 1024);
      const SmemDesc dDS_mn = sw128_desc_words(sbase + C::kOffDS, C::kBlockBytes, 1024);
      if (issuer_a) {
        auto issue_s = [&](int s) {   // S^T = K Q^T -> X
          const SmemDesc dq = desc_step(dQ_k, (s & 1) * C::kQTileBytes);
#pragma unroll 1
          for (int kk = 0; kk < DH / 16; ++kk) {
            const uint32_t off = (kk >> 2) * C::kBlockBytes + (kk & 3) * 32;
            umma_ss_we(tmem + C::kTX, desc_step(dK_k, off), desc_step(dq, off), kIdS, kk > 0 ? 1u : 0u);
          }
          umma_commit_we(bar(C::kBarSFull));
        };
        auto issue_dp = [&]() {  // dP^T = V dO^T -> Y
#pragma unroll 1
          for (int kk = 0; kk < DV / 16; ++kk) {
            const uint32_t off = (kk >> 2) * C::kBlockBytes + (kk & 3) * 32;
            umma_ss_we(tmem + C::kTY, desc_step(dV_k, off), desc_step(dDO_k, off), kIdDP, kk > 0 ? 1u : 0u);
          }
          umma_commit_we(bar(C::kBarDPFull));
        };
        // The two score warpgroups leave P^T for queries [0,64) in columns
        // [0,32) and for queries [64,128) in columns [64,96) of X.
        auto half_col = [](int kk) { return static_cast<uint32_t>(64 * (kk >> 2) + 8 * (kk & 3)); };
        if (ok) ok = wait_all(C::kBarQFull + 0, 0);
        if (ok) {
          tc_fence_after_sync();
          issue_s(0);
        }
        if (ok) ok = wait_all(C::kBarDOFull, 0);
        if (ok) ok = wait_all(C::kBarV16, 0);
        if (ok) {
          tc_fence_after_sync();
          issue_dp();
        }
        for (int s = 0; s < total && ok; ++s) {
          ok = wait_all(C::kBarPReady, static_cast<uint32_t>(s & 1));
          if (!ok) break;
          tc_fence_after_sync();
#pragma unroll 1
          for (int kk = 0; kk < kTileM / 16; ++kk)
            umma_ts_we(tmem + C::kTdV, tmem + C::kTX + half_col(kk), desc_step(dDO_mn, kk * 2048), kIdDV,
                      (s > 0 || kk > 0) ? 1u : 0u);
          umma_commit_we(bar(C::kBarDOEmpty));   // dP(s) and dV(s) were dO(s)'s only readers
          if (s + 1 < total) {
            ok = wait_all(C::kBarQFull + ((s + 1) & 1), static_cast<uint32_t>(((s + 1) >> 1) & 1));
            if (!ok) break;
            tc_fence_after_sync();
            issue_s(s + 1);
            ok = wait_all(C::kBarDOFull, static_cast<uint32_t>((s + 1) & 1));
            if (ok) ok = wait_all(C::kBarDQFree, static_cast<uint32_t>(s & 1));
            if (ok) ok = wait_all(C::kBarDKDone, static_cast<uint32_t>(s & 1));
            if (!ok) break;
            tc_fence_after_sync();
            issue_dp();
          }
        }
      } else {
        for (int s = 0; s < total && ok; ++s) {
          ok = wait_all(C::kBarDSReady, static_cast<uint32_t>(s & 1));
          if (!ok) break;
          tc_fence_after_sync();
          // dQ(s) first, into Y (the score warps have read dP^T out of it),
          // so that its read-out overlaps dK(s); both take dS from the
          // shared-memory buffer, as the MN-major (dQ) and the K-major (dK)
          // view of the same swizzled tile.
#pragma unroll 1
          for (int kk = 0; kk < kTileN / 16; ++kk)
            umma_ss_we(tmem + C::kTY, desc_step(dDS_mn, kk * 2048), desc_step(dK_mn, kk * 2048), kIdDQ,
                      kk > 0 ? 1u : 0u);
          umma_commit_we(bar(C::kBarDQFull));
#pragma unroll 1
          for (int kk = 0; kk < kTileM / 16; ++kk)
            umma_ss_we(tmem + C::kTdK, desc_step(dDS_k, (kk >> 2) * C::kBlockBytes + (kk & 3) * 32),
                      desc_step(dQ_mn, (s & 1) * C::kQTileBytes + kk * 2048), kIdDK, (s > 0 || kk > 0) ? 1u : 0u);
          umma_commit_we(bar(C::kBarQEmpty + (s & 1)));
          umma_commit_we(bar(C::kBarDKDone));
        }
      }
      if (ok) umma_commit_we(bar(C::kBarDKDV));
      int no_abort = 0;
      umma_commit_we(bar(C::kBarDrain));
      mbar_wait(bar(C::kBarDrain), 0, &no_abort, limit);
    }
    __syncwarp();
  } else if (warp >= 4 && warp < 12) {
    // =========================== score warpgroups =======================
    // Two warpgroups: h = 0 takes query columns [0, 64), h = 1 [64, 128);
    // in both, thread = key row = TMEM lane.
    setmaxnreg_to<C::kRegsScore, C::kRegsLaunch>();
    const int h = static_cast<int>(warp - 4) / 4;
    const uint32_t quad = warp & 3;
    const int jj = static_cast<int>(quad * 32 + lane);
    const int tid = static_cast<int>(threadIdx.x) - 128 - 128 * h;
    const int64_t j = j0 + jj;
    const bool row_masked = j >= klen;
    const uint32_t lane_base = (quad * 32u) << 16;
    const uint32_t tX = tmem + lane_base + C::kTX;
    const uint32_t tY = tmem + lane_base + C::kTY;
    uint8_t* ds_row = smem + C::kOffDS + h * C::kBlockBytes + jj * 128;
    bool ok = *abort_flag == 0 && total > 0;
    if (ok && h == 0) {
      // ---- the bound on |dS| for this CTA (CtaScale) ----
      // From the bf16 V tile's row norms (the read-out warps re-encode it
      // only after this reduction is published) and every step's tile
      // maxima.
      ok = wait_all(C::kBarKV, 0);
      float vn2 = 0.f;
      if (ok && !row_masked) {
#pragma unroll
        for (int c = 0; c < DV / 64; ++c) {
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const uint4 u = *reinterpret_cast<const uint4*>(smem + C::kOffV + c * C::kBlockBytes + jj * 128 + q * 16);
            const uint32_t wv[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              vn2 = fmaf(bf16_lo(wv[k]), bf16_lo(wv[k]), vn2);
              vn2 = fmaf(bf16_hi(wv[k]), bf16_hi(wv[k]), vn2);
            }
          }
        }
      }
      float mv = sqrtf(vn2), mdo = 0.f, md = 0.f;
      for (int idx = tid; idx < total; idx += 128) {
        const int bhq = b * p.sh.Hq + step_head(idx);
        const float4 t = p.tilemax[static_cast<int64_t>(bhq) * p.nqt + step_q0(idx) / kTileM];
        mdo = fmaxf(mdo, t.x);
        md = fmaxf(md, t.y);
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        mv = fmaxf(mv, __shfl_xor_sync(0xffffffffu, mv, off));
        mdo = fmaxf(mdo, __shfl_xor_sync(0xffffffffu, mdo, off));
        md = fmaxf(md, __shfl_xor_sync(0xffffffffu, md, off));
      }
      if (lane == 0) {
        red_s[4 * quad] = mv;
        red_s[4 * quad + 1] = mdo;
        red_s[4 * quad + 2] = md;
      }
      mbar_arrive(bar(C::kBarScale));
    }
    CtaScale cs{};
    const float2 qo = ok ? group_exps() : make_float2(0.f, 0.f);
    if (ok) ok = wait_all(C::kBarScale, 0);
    // The CTA's multipliers (CtaScale): the scores come out of S^T = K16
    // Q16^T as 2^(k + q) S_raw, so P = exp2(S_acc sl2 - LSE log2e) with
    // sl2 = scale log2e 2^-(k + q); and dS' = 2^g dS =
    // P (dP_acc cp + (-D) dmul) with cp = 2^(g - o - v), dmul = 2^g.
    float sl2 = p.scale_log2, cp = 1.f, dmul = 1.f;
    // The weights P of this thread's 64 columns, kept in fp32 from the P pass
    // for the dS pass (the fp16 copy goes to tensor memory for dV).
    float pf[64];
    // This thread's -LSE log2(e) and -D entries (query q0 + 64h + tid, for
    // tid < 64) of a step, loaded one step ahead so the global latency is
    // off the critical path.  Both are kept negated so that one paired
    // fused multiply-add forms x sl2 - LSE log2(e) and dP_acc cp - D dmul.
    auto load_row_terms = [&](int s, float& nlse2, float& nd) {
      const int64_t i = static_cast<int64_t>(step_q0(s)) + 64 * h + tid;
      // Query rows past the sequence get LSE = -inf: their weights P, and so
      // their dS and contributions to dK, dV, dQ, are exactly 0.
      const bool in = tid < 64 && i < nq_b;
      const int64_t r = in ? q_vec(PACKED, p.lay, p.sh.Hq, p.sh.n_q, b, step_head(s), i) : 0;
      nlse2 = in ? -p.LSE[r] * kLog2e : -INFINITY;
      nd = in ? -p.D[r] : 0.f;
    };
    // Each warpgroup reads only its own 64 LSE/D entries, written by its own
    // threads tid < 64, so the two warpgroups never wait for each other
    // here: a 128-thread named barrier publishes the entries of step s
    // before its passes, and a second one ends every reader of step s
    // before the entries of step s+1 overwrite them.  Every thread passes
    // both barriers of every step, even after an abort (the step's work is
    // then skipped), so no warp can be left waiting at one.
    float lse_next = 0.f, d_next = 0.f;
    if (ok) load_row_terms(0, lse_next, d_next);
    if (ok) ok = wait_all(C::kBarK16, 0);   // the read-out warps publish the K exponent with it
    if (ok) {
      cs = cta_scale(red_s, qo);
      const int kexp = static_cast<int>(red_s[C::kRedKExp]);
      sl2 = p.scale_log2 * exp2_int(-kexp - cs.q);
      cp = exp2_int(cs.g - cs.o - cs.v);
      dmul = exp2_int(cs.g);
      if (tid < 64) {
        lse_s[64 * h + tid] = lse_next;
        dd_s[64 * h + tid] = d_next * dmul;
      }
      if (total > 1) load_row_terms(1, lse_next, d_next);
    }
    const uint32_t wg_bar = 1 + static_cast<uint32_t>(h);
    for (int s = 0; s < total; ++s) {
      named_bar_sync(wg_bar, 128);
      do {
      if (!ok) break;
      const int q0 = step_q0(s);
      // Column c (query q0 + c) is visible iff this key row is inside
      // kv_len and, when causal, q0 + c >= j - offset.
      const int64_t cmin64 = p.mask.causal ? (j - causal_offset(p.mask, b) - q0) : INT64_MIN / 2;
      const int cmin = cmin64 > kTileM ? kTileM + 1 : (cmin64 < -1 ? -1 : static_cast<int>(cmin64));
      // Packed sequences: columns c >= cmax are query rows of the next
      // sequence; their weights and dS are set to 0 outright.  (In the padded
      // layout the rows past n_q read as zeros and carry LSE = -inf.)
      const int64_t cmax64 = nq_b - q0;
      const int cmax = (!PACKED || cmax64 > kTileM) ? kTileM : static_cast<int>(cmax64);
      const bool need_mask =
          __any_sync(0xffffffffu, row_masked || cmin > 64 * h || (PACKED && cmax < 64 * h + 64));
      ok = wait_all(C::kBarSFull, static_cast<uint32_t>(s & 1));
      if (!ok) break;
      tc_fence_after_sync();
      // P pass: this half's 64 scores in registers (two loads, one wait).
      // P^T (fp16) goes into X over the columns already read; the fp32
      // weights stay in registers for the dS pass (no fp16 unpacking there:
      // 1.4-1.9 % of the main kernel on c3 and c5 in same-box runs).
      {
        uint32_t sa[32], sb[32];
        tmem_ld32_nowait(tX + 64 * h, sa);
        tmem_ld32_nowait(tX + 64 * h + 32, sb);
        tmem_wait_ld32(sa);
        tmem_wait_ld32(sb);
#pragma unroll
        for (int cq = 0; cq < 4; ++cq) {
          float nl[16];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const float4 v = *reinterpret_cast<const float4*>(lse_s + 64 * h + cq * 16 + 4 * q);
            nl[4 * q] = v.x;
            nl[4 * q + 1] = v.y;
            nl[4 * q + 2] = v.z;
            nl[4 * q + 3] = v.w;
          }
          uint32_t w[8];
#pragma unroll
          for (int k = 0; k < 16; k += 2) {
            const int c = 64 * h + cq * 16 + k;
            const int r = (cq & 1) * 16 + k;
            const float s0 = __uint_as_float(cq < 2 ? sa[r] : sb[r]);
            const float s1 = __uint_as_float(cq < 2 ? sa[r + 1] : sb[r + 1]);
            float x0, x1;
            ffma2(x0, x1, s0, s1, sl2, sl2, nl[k], nl[k + 1]);
            if (need_mask) {
              x0 = (!row_masked && c >= cmin && (!PACKED || c < cmax)) ? x0 : -INFINITY;
              x1 = (!row_masked && c + 1 >= cmin && (!PACKED || c + 1 < cmax)) ? x1 : -INFINITY;
            }
            const float p0 = fast_exp2(x0), p1 = fast_exp2(x1);
            w[k >> 1] = pack_f16x2(p0, p1);
            pf[cq * 16 + k] = p0;
            pf[cq * 16 + k + 1] = p1;
          }
          tmem_st8_nowait(tX + 64 * h + cq * 8, w);
        }
        tmem_wait_st();
      }
      tc_fence_before_sync();
      mbar_arrive(bar(C::kBarPReady));
      ok = wait_all(C::kBarDPFull, static_cast<uint32_t>(s & 1));
      if (!ok) break;
      tc_fence_after_sync();
      // dS pass: dS' = dS 2^g (CtaScale) as fp16 into this half's block of
      // the dS buffer (for dQ and dK).
      {
        uint32_t da[32], db[32];
        tmem_ld32_nowait(tY + 64 * h, da);
        tmem_ld32_nowait(tY + 64 * h + 32, db);
        tmem_wait_ld32(da);
        tmem_wait_ld32(db);
#pragma unroll
        for (int cq = 0; cq < 4; ++cq) {
          float nd[16];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const float4 v = *reinterpret_cast<const float4*>(dd_s + 64 * h + cq * 16 + 4 * q);
            nd[4 * q] = v.x;
            nd[4 * q + 1] = v.y;
            nd[4 * q + 2] = v.z;
            nd[4 * q + 3] = v.w;
          }
          uint32_t w[8];
#pragma unroll
          for (int k = 0; k < 16; k += 2) {
            const int c = 64 * h + cq * 16 + k;
            const int r = (cq & 1) * 16 + k;
            const float g0 = __uint_as_float(cq < 2 ? da[r] : db[r]);
            const float g1 = __uint_as_float(cq < 2 ? da[r + 1] : db[r + 1]);
            float t0, t1, d0, d1;
            ffma2(t0, t1, g0, g1, cp, cp, nd[k], nd[k + 1]);
            fmul2(d0, d1, pf[cq * 16 + k], pf[cq * 16 + k + 1], t0, t1);
            if (need_mask) {
              d0 = (!row_masked && c >= cmin && (!PACKED || c < cmax)) ? d0 : 0.f;
              d1 = (!row_masked && c + 1 >= cmin && (!PACKED || c + 1 < cmax)) ? d1 : 0.f;
            }
            w[k >> 1] = pack_f16x2(d0, d1);
          }
          // dS (queries contiguous per key row) for the dQ = dS K and
          // dK = dS^T Q products: this half's 64 queries fill one 128-byte
          // row of its block, the 16-byte chunk index XOR-swizzled with the
          // key row.
#pragma unroll
          for (int v = 0; v < 2; ++v) {
            const int chunk = cq * 2 + v;
            *reinterpret_cast<uint4*>(ds_row + ((chunk ^ (jj & 7)) * 16)) =
                make_uint4(w[4 * v], w[4 * v + 1], w[4 * v + 2], w[4 * v + 3]);
          }
        }
      }
      fence_proxy_async_smem();
      tc_fence_before_sync();
      mbar_arrive(bar(C::kBarDSReady));
      } while (false);
      named_bar_sync(wg_bar, 128);
      if (ok && tid < 64 && s + 1 < total) {
        lse_s[64 * h + tid] = lse_next;
        dd_s[64 * h + tid] = d_next * dmul;
      }
      if (ok && s + 2 < total) load_row_terms(s + 2, lse_next, d_next);
    }
  } else if (warp >= 12) {
    // ======== fp16 re-encoding of K, dQ read-out, dK/dV epilogue ========
    setmaxnreg_to<C::kRegsAux, C::kRegsLaunch>();
    const uint32_t quad = warp & 3;
    const int row = static_cast<int>(quad * 32 + lane);
    const int tid2 = static_cast<int>(threadIdx.x) - 384;
    const uint32_t lane_base = (quad * 32u) << 16;
    bool ok = *abort_flag == 0;
    uint32_t rr[32];
    CtaScale cs{};
    int kexp = 0;
    const float2 qo = (ok && total > 0) ? group_exps() : make_float2(0.f, 0.f);
    if (total > 0) {
      // K and V once, as fp16 x 2^k and x 2^v (CtaScale): rows in
      // [kv_len, n_k) hold caller memory that may be anything (even NaN) and
      // become zeros -- their dS entries are 0, but 0 * NaN would still
      // poison dQ.  Rows at or beyond n_k arrive as zeros from the TMA
      // bounds check.  K first (the first product needs it): the whole tile
      // is held in registers while the four warps agree on its largest
      // magnitude; V once the score warps have published the reduction its
      // exponent comes from.
      constexpr int kKc = C::kKTileBytes / 16 / 128;
      uint4* kt = reinterpret_cast<uint4*>(smem + C::kOffK);
      auto tile_row = [](int k) { return (k % (C::kBlockBytes / 16)) / 8; };   // 8 chunks per 128-byte row
      if (ok) ok = wait_all(C::kBarKV, 0);
      uint32_t km = 0u;
      if (ok) {
#pragma unroll 8
        for (int i = 0; i < kKc; ++i) {
          const uint4 u = kt[tid2 + 128 * i];
          if (j0 + tile_row(tid2 + 128 * i) < klen) km = bf16_absmax_fold(km, u);
        }
      }
      float kmax = bf16_absmax_value(km);
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) kmax = fmaxf(kmax, __shfl_xor_sync(0xffffffffu, kmax, off));
      if (lane == 0) red_s[C::kRedK + quad] = kmax;
      named_bar_sync(3, 128);   // passed by all four warps, even after an abort
      kmax = fmaxf(fmaxf(red_s[C::kRedK], red_s[C::kRedK + 1]), fmaxf(red_s[C::kRedK + 2], red_s[C::kRedK + 3]));
      kexp = f16_tile_exponent(kmax);
      if (kexp == kExpZero) kexp = 0;
      if (ok) {
        const float ks = exp2_int(kexp);
        for (int i0 = 0; i0 < kKc; i0 += 8) {
          uint4 kv[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) kv[i] = kt[tid2 + 128 * (i0 + i)];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int k = tid2 + 128 * (i0 + i);
            kt[k] = (j0 + tile_row(k) >= klen) ? make_uint4(0u, 0u, 0u, 0u) : bf16x8_to_f16x8_scaled(kv[i], ks);
          }
        }
        if (tid2 == 0) red_s[C::kRedKExp] = static_cast<float>(kexp);
        fence_proxy_async_smem();
        mbar_arrive(bar(C::kBarK16));
      }
      if (ok) ok = wait_all(C::kBarScale, 0);
      if (ok) {
        cs = cta_scale(red_s, qo);
        if (tid2 == 0 && (f16_saturates(kmax, kexp) || f16_saturates(cs.mv, cs.v) || cs.overflow))
          record_status(p.status, ATTN_ERR_RANGE);
        // V in place, eight loads in flight per thread before their stores.
        const float vs = exp2_int(cs.v);
        uint4* vt = reinterpret_cast<uint4*>(smem + C::kOffV);
        for (int i0 = 0; i0 < C::kVTileBytes / 16 / 128; i0 += 8) {
          uint4 v[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) v[i] = vt[tid2 + 128 * (i0 + i)];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int k = tid2 + 128 * (i0 + i);
            vt[k] = (j0 + tile_row(k) >= klen) ? make_uint4(0u, 0u, 0u, 0u) : bf16x8_to_f16x8_scaled(v[i], vs);
          }
        }
        fence_proxy_async_smem();
        mbar_arrive(bar(C::kBarV16));
      }
    }
    // dQ read-out: each warp takes its 32 query rows of the tile (in Y) into
    // registers a 64-column round at a time and releases Y after the last
    // round's loads; it scales them back by 2^-(g + k) (dQ_acc = dS' K16,
    // CtaScale) and stages them as 32 x 32 fp32 boxes in the 128-byte swizzle
    // pattern (conflict-free stores), and one lane adds the boxes into the
    // fp32 accumulator with TMA reduce-add, a round at a time, the staging
    // memory being reused once a round's boxes have been read.  Rows past
    // n_q are clipped by the tensor map.
    const uint32_t tY = tmem + lane_base + C::kTY;
    auto stage_box = [&](uint8_t* dst_box, const uint32_t (&v)[32], float inv) {
      uint8_t* dst = dst_box + lane * 128;
#pragma unroll
      for (int c = 0; c < 8; ++c)
        *reinterpret_cast<float4*>(dst + ((c ^ (lane & 7)) * 16)) =
            make_float4(__uint_as_float(v[4 * c]) * inv, __uint_as_float(v[4 * c + 1]) * inv,
                        __uint_as_float(v[4 * c + 2]) * inv, __uint_as_float(v[4 * c + 3]) * inv);
    };
    auto reduce_round = [&](uint8_t* wstage, int first_box, int row0, int head) {
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0 && row0 < nq_b) {
        // (Rows of the box past the sequence hold zeros: adding them is a
        // no-op on whatever rows lie there.)
        const TmaYZ yz = q_tma(PACKED, p.lay, p.sh.Hq, b, head, row0);
#pragma unroll
        for (int bx = 0; bx < C::kDQBoxesPerRound; ++bx)
          tma_reduce_add_3d(&tmdQ, smem_u32(wstage + bx * C::kDQBoxBytes), (first_box + bx) * C::kDQBoxCols, yz.y,
                            yz.z);
        bulk_commit_group();
      }
    };
    // The staging memory is rewritten only once the reduce-adds already
    // issued from it have read it (the last round of a step completes while
    // the next step's MMAs run).
    auto staging_free = [&]() {
      if (lane == 0) bulk_wait_group_read0();
      __syncwarp();
    };
    const float inv = exp2_int(-cs.g - kexp);
    for (int s = 0; s < total && ok; ++s) {
      const int head = step_head(s);
      const int q0 = step_q0(s);
      const int row0 = q0 + static_cast<int>(quad) * 32;
      ok = wait_all(C::kBarDQFull, static_cast<uint32_t>(s & 1));
      if (!ok) break;
      tc_fence_after_sync();
      uint8_t* wstage = smem + C::kOffStage + quad * C::kDQWarpStage;
      // A round at a time: two 32-column loads behind one wait; Y is handed
      // back after the last round's loads.
#pragma unroll
      for (int rd = 0; rd < C::kDQRounds; ++rd) {
        uint32_t v[C::kDQBoxesPerRound][32];
#pragma unroll
        for (int bx = 0; bx < C::kDQBoxesPerRound; ++bx)
          tmem_ld32_nowait(tY + (rd * C::kDQBoxesPerRound + bx) * C::kDQBoxCols, v[bx]);
#pragma unroll
        for (int bx = 0; bx < C::kDQBoxesPerRound; ++bx) tmem_wait_ld32(v[bx]);
        if (rd + 1 == C::kDQRounds) {
          tc_fence_before_sync();
          mbar_arrive(bar(C::kBarDQFree));
        }
        staging_free();
#pragma unroll
        for (int bx = 0; bx < C::kDQBoxesPerRound; ++bx) stage_box(wstage + bx * C::kDQBoxBytes, v[bx], inv);
        reduce_round(wstage, rd * C::kDQBoxesPerRound, row0, head);
      }
      __syncwarp();
    }
    if (lane == 0) bulk_wait_group0();
    if (ok && total > 0) {
      ok = wait_all(C::kBarDKDV, 0);
      tc_fence_after_sync();
    }
    if constexpr (SPLIT) {
     if (ok) {
      // This CTA's share of dK, dV, in fp32, added into the split's sums
      // (dK turned back by the rotary first: the turn is linear).  The
      // tensor-memory loads are warp-collective: every lane takes part, and
      // only the rows inside the sequence are added.
      const int64_t j = j0 + row;
      const bool in = j < k_row_end;
      if (total > 0) {
        const float dk_scale = p.scale * exp2_int(-cs.g - cs.q);
        const float dv_scale = exp2_int(-cs.o);
        const int64_t arow = PACKED ? (static_cast<int64_t>(p.lay.cu_k[b]) + j) * p.sh.Hkv + hkv
                                    : (static_cast<int64_t>(b) * p.sh.Hkv + hkv) * p.sh.n_k + j;
        int32_t kpos = 0;
        if constexpr (ROPE) kpos = in ? p.rot.pos[k_token(PACKED, p.lay, p.sh.n_k, b, j)] : 0;
#pragma unroll 1
        for (int cc = 0; cc < DH / 32; ++cc) {
          tmem_ld32(tmem + lane_base + C::kTdK + cc * 32, rr);
          float y[32];
#pragma unroll
          for (int k = 0; k < 32; ++k) y[k] = __uint_as_float(rr[k]) * dk_scale;
          if constexpr (ROPE) {
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
              float wh[4], wl[4];
              rope_freqs4(p.rot.w_hi, p.rot.w_lo, 4 * cc + q4, wh, wl);
              float4 t0, t1;
              rope_angles4(kpos, wh, wl, t0, t1);
              rope_transpose(t0, t1);
              const float cs4[4] = {t0.x, t0.z, t1.x, t1.z}, sn4[4] = {t0.y, t0.w, t1.y, t1.w};
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                const int k = 8 * q4 + 2 * q;
                rot_block(y[k], y[k + 1], cs4[q], sn4[q], y[k], y[k + 1]);
              }
            }
          }
          float* dst = p.dKacc + arow * DH + cc * 32;
          if (in) {
#pragma unroll
            for (int c = 0; c < 8; ++c)
              asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(dst + 4 * c), "f"(y[4 * c]),
                           "f"(y[4 * c + 1]), "f"(y[4 * c + 2]), "f"(y[4 * c + 3])
                           : "memory");
          }
        }
#pragma unroll 1
        for (int cc = 0; cc < DV / 32; ++cc) {
          tmem_ld32(tmem + lane_base + C::kTdV + cc * 32, rr);
          float* dst = p.dVacc + arow * DV + cc * 32;
          if (in) {
#pragma unroll
            for (int c = 0; c < 8; ++c)
              asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(dst + 4 * c),
                           "f"(__uint_as_float(rr[4 * c]) * dv_scale), "f"(__uint_as_float(rr[4 * c + 1]) * dv_scale),
                           "f"(__uint_as_float(rr[4 * c + 2]) * dv_scale),
                           "f"(__uint_as_float(rr[4 * c + 3]) * dv_scale)
                           : "memory");
          }
        }
      }
     }
    } else if (ok) {
      const int64_t j = j0 + row;
      const bool in = j < k_row_end;
      uint4* dk = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.dK) +
                                           strided_off(PACKED, p.lay.sdk, p.sh.Hkv, p.lay.cu_k[b], b, hkv, j));
      uint4* dv = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.dV) +
                                           strided_off(PACKED, p.lay.sdv, p.sh.Hkv, p.lay.cu_k[b], b, hkv, j));
      const float dk_scale = p.scale * exp2_int(-cs.g - cs.q);   // dK_acc = 2^(g + q) dS^T Q (CtaScale)
      const float dv_scale = exp2_int(-cs.o);                    // dV_acc = 2^o P^T dO
      // Rotary: the accumulated gradient is that of the rotated key; the
      // key's own gradient is it turned back by the key's angles (the
      // transpose of the rotation), formed here per 4-block chunk.
      int32_t kpos = 0;
      if constexpr (ROPE) kpos = in ? p.rot.pos[k_token(PACKED, p.lay, p.sh.n_k, b, j)] : 0;
      // (With the rotary the chunks stay rolled: each unrolled chunk would
      // carry its own copy of the angle arithmetic.)
      constexpr int kDkUnroll = ROPE ? 1 : DH / 32;
#pragma unroll kDkUnroll
      for (int cc = 0; cc < DH / 32; ++cc) {
        uint32_t w[16];
        if (total > 0) {
          tmem_ld32(tmem + lane_base + C::kTdK + cc * 32, rr);
          if constexpr (ROPE) {
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {   // chunk 4 cc + q4: columns 32 cc + 8 q4 ..
              float wh[4], wl[4];
              rope_freqs4(p.rot.w_hi, p.rot.w_lo, 4 * cc + q4, wh, wl);
              float4 t0, t1;
              rope_angles4(kpos, wh, wl, t0, t1);
              rope_transpose(t0, t1);
              const float cs4[4] = {t0.x, t0.z, t1.x, t1.z}, sn4[4] = {t0.y, t0.w, t1.y, t1.w};
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                const int k = 8 * q4 + 2 * q;
                float y0, y1;
                rot_block(__uint_as_float(rr[k]) * dk_scale, __uint_as_float(rr[k + 1]) * dk_scale, cs4[q], sn4[q],
                          y0, y1);
                w[k >> 1] = pack_bf16x2(y0, y1);
              }
            }
          } else {
#pragma unroll
            for (int k = 0; k < 32; k += 2)
              w[k >> 1] = pack_bf16x2(__uint_as_float(rr[k]) * dk_scale, __uint_as_float(rr[k + 1]) * dk_scale);
          }
        } else {
#pragma unroll
          for (int k = 0; k < 16; ++k) w[k] = 0u;
        }
        if (in) {
#pragma unroll
          for (int v = 0; v < 4; ++v) dk[cc * 4 + v] = make_uint4(w[4 * v], w[4 * v + 1], w[4 * v + 2], w[4 * v + 3]);
        }
      }
#pragma unroll
      for (int cc = 0; cc < DV / 32; ++cc) {
        uint32_t w[16];
        if (total > 0) {
          tmem_ld32(tmem + lane_base + C::kTdV + cc * 32, rr);
#pragma unroll
          for (int k = 0; k < 32; k += 2)
            w[k >> 1] = pack_bf16x2(__uint_as_float(rr[k]) * dv_scale, __uint_as_float(rr[k + 1]) * dv_scale);
        } else {
#pragma unroll
          for (int k = 0; k < 16; ++k) w[k] = 0u;
        }
        if (in) {
#pragma unroll
          for (int v = 0; v < 4; ++v) dv[cc * 4 + v] = make_uint4(w[4 * v], w[4 * v + 1], w[4 * v + 2], w[4 * v + 3]);
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

// Per-tile work of the backward preprocess, for a 128-row query tile:
//   D_i = sum_l dO_il (O_il + O_lo_il)   (O_lo may be absent),
//   tilemax = (max_i ||dO_i||_2, max_i |D_i|, e_Q, e_dO) over the tile's rows,
// the tile's rows of the fp32 dQ accumulator are zeroed, and its rows of Q
// and dO are re-encoded as fp16 for the main kernel, scaled by 2^e_Q and
// 2^e_dO (f16range.cuh: the exponents come from the tile's largest
// magnitudes, so the re-encoding is exact whatever the inputs' scale).  The
// whole tile's Q and dO therefore stay in registers until the block has
// reduced its maxima.  In the D pass each row has DV/8 consecutive threads,
// one 16-byte chunk each, so every warp load covers whole rows.
// row_at(rr) is the workspace row of the tile's row rr (the contiguous
// layout of Q), d_at(rr) its index in D, and user_at(s, rr) its element
// offset in a user tensor with strides s.  ROPE: Q is the rotated query,
// each row turned by the angles of its token tok_at(rr) (positions and
// frequencies rot) and rounded to bf16 as the forward's rotation rounds it.
template <int DV, int DH, bool ROPE, class RowAt, class DAt, class UserAt, class TokAt>
__device__ __forceinline__ void bwd_prep_tile(int rows_here, const RowAt& row_at, const DAt& d_at,
                                              const UserAt& user_at, const TokAt& tok_at, const RotaryAngles& rot,
                                              const TensorStrides& sq,
                                              const TensorStrides& so, const TensorStrides& sdo,
                                              const uint4* __restrict__ Q, const uint4* __restrict__ O,
                                              const uint4* __restrict__ O_lo, const uint4* __restrict__ dO,
                                              float* __restrict__ D, float4* __restrict__ tm,
                                              float4* __restrict__ dQacc, uint4* __restrict__ Q16,
                                              uint4* __restrict__ dO16, unsigned int* status) {
  constexpr int kTpr = DV / 8;                 // threads per row in the D pass
  constexpr int kRows = 256 / kTpr;            // rows per pass
  constexpr int kPasses = kTileM / kRows;
  constexpr int kBatch = 2;                    // passes whose O loads are in flight together
  static_assert(kPasses % kBatch == 0, "pass count");
  constexpr int kQ = kTileM * (DH / 8) / 256, kZ = kTileM * (DH / 4) / 256;
  __shared__ float red[4][8];
  const int c = static_cast<int>(threadIdx.x) % kTpr, r0 = static_cast<int>(threadIdx.x) / kTpr;
  // Q first: its loads stay in flight through the D pass.
  uint4 q[kQ];
#pragma unroll
  for (int j = 0; j < kQ; ++j) {
    const int k = j * 256 + static_cast<int>(threadIdx.x), rr = k / (DH / 8);
    q[j] = rr < rows_here ? Q[user_at(sq, rr) / 8 + k % (DH / 8)] : make_uint4(0u, 0u, 0u, 0u);
  }
  if constexpr (ROPE) {
    // A thread keeps one chunk (256 is a multiple of the row's DH / 8
    // chunks), so its four frequencies serve all its rows; the positions are
    // requested right behind the rows, which are turned before the D pass.
    float wh[4], wl[4];
    rope_freqs4(rot.w_hi, rot.w_lo, static_cast<int>(threadIdx.x) % (DH / 8), wh, wl);
    int32_t pos[kQ];
#pragma unroll
    for (int j = 0; j < kQ; ++j) {
      const int rr = (j * 256 + static_cast<int>(threadIdx.x)) / (DH / 8);
      pos[j] = rr < rows_here ? rot.pos[tok_at(rr)] : 0;
    }
#pragma unroll
    for (int j = 0; j < kQ; ++j) {
      const int rr = (j * 256 + static_cast<int>(threadIdx.x)) / (DH / 8);
      if (rr < rows_here) {
        float4 t0, t1;
        rope_angles4(pos[j], wh, wl, t0, t1);
        q[j] = rot_bf16x8(q[j], t0, t1);
      }
    }
  }
  float mn = 0.f, md = 0.f;
  uint32_t gmax = 0u, qmax = 0u;
  uint4 g[kPasses];
#pragma unroll
  for (int p0 = 0; p0 < kPasses; p0 += kBatch) {
    uint4 a[kBatch], lo[kBatch];
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int rr = (p0 + u) * kRows + r0;
      a[u] = g[p0 + u] = lo[u] = make_uint4(0u, 0u, 0u, 0u);
      if (rr < rows_here) {
        const int64_t at = user_at(so, rr) / 8 + c;
        a[u] = O[at];
        g[p0 + u] = dO[user_at(sdo, rr) / 8 + c];
        if (O_lo) lo[u] = O_lo[at];
      }
    }
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int rr = (p0 + u) * kRows + r0;
      const uint4 gu = g[p0 + u];
      const uint32_t aw[4] = {a[u].x, a[u].y, a[u].z, a[u].w};
      const uint32_t gw[4] = {gu.x, gu.y, gu.z, gu.w};
      const uint32_t lw[4] = {lo[u].x, lo[u].y, lo[u].z, lo[u].w};
      float acc = 0.f, nrm = 0.f;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float g0 = bf16_lo(gw[k]), g1 = bf16_hi(gw[k]);
        acc = fmaf(bf16_lo(aw[k]) + bf16_lo(lw[k]), g0, acc);
        acc = fmaf(bf16_hi(aw[k]) + bf16_hi(lw[k]), g1, acc);
        nrm = fmaf(g0, g0, nrm);
        nrm = fmaf(g1, g1, nrm);
      }
      gmax = bf16_absmax_fold(gmax, gu);
#pragma unroll
      for (int off = kTpr / 2; off > 0; off >>= 1) {
        acc += __shfl_xor_sync(0xffffffffu, acc, off);
        nrm += __shfl_xor_sync(0xffffffffu, nrm, off);
      }
      if (rr < rows_here) {
        if (c == 0) D[d_at(rr)] = acc;
        mn = fmaxf(mn, sqrtf(nrm));
        md = fmaxf(md, fabsf(acc));
      }
    }
  }
#pragma unroll
  for (int j = 0; j < kQ; ++j) qmax = bf16_absmax_fold(qmax, q[j]);
  // Block maxima: row norms and |D| agree across a row's kTpr lanes already;
  // the magnitude maxima differ per thread.
  float gm = bf16_absmax_value(gmax), qm = bf16_absmax_value(qmax);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    if (off >= kTpr) {
      mn = fmaxf(mn, __shfl_xor_sync(0xffffffffu, mn, off));
      md = fmaxf(md, __shfl_xor_sync(0xffffffffu, md, off));
    }
    gm = fmaxf(gm, __shfl_xor_sync(0xffffffffu, gm, off));
    qm = fmaxf(qm, __shfl_xor_sync(0xffffffffu, qm, off));
  }
  if ((threadIdx.x & 31) == 0) {
    red[0][threadIdx.x >> 5] = mn;
    red[1][threadIdx.x >> 5] = md;
    red[2][threadIdx.x >> 5] = gm;
    red[3][threadIdx.x >> 5] = qm;
  }
  __syncthreads();
  float x = 0.f, y = 0.f;
  gm = qm = 0.f;
#pragma unroll
  for (int w = 0; w < 8; ++w) {
    x = fmaxf(x, red[0][w]);
    y = fmaxf(y, red[1][w]);
    gm = fmaxf(gm, red[2][w]);
    qm = fmaxf(qm, red[3][w]);
  }
  const int eq = f16_tile_exponent(qm), eo = f16_tile_exponent(gm);
  if (threadIdx.x == 0) {
    *tm = make_float4(x, y, static_cast<float>(eq), static_cast<float>(eo));
    if (f16_saturates(qm, eq) || f16_saturates(gm, eo)) record_status(status, ATTN_ERR_RANGE);
  }
  const float sco = exp2_int(eo == kExpZero ? 0 : eo), scq = exp2_int(eq == kExpZero ? 0 : eq);
#pragma unroll
  for (int p0 = 0; p0 < kPasses; ++p0) {
    const int rr = p0 * kRows + r0;
    if (rr < rows_here) dO16[row_at(rr) * (DV / 8) + c] = bf16x8_to_f16x8_scaled(g[p0], sco);
  }
#pragma unroll
  for (int j = 0; j < kZ; ++j) {
    const int k = j * 256 + static_cast<int>(threadIdx.x), rr = k / (DH / 4);
    if (rr < rows_here) dQacc[row_at(rr) * (DH / 4) + k % (DH / 4)] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
#pragma unroll
  for (int j = 0; j < kQ; ++j) {
    const int k = j * 256 + static_cast<int>(threadIdx.x), rr = k / (DH / 8);
    if (rr < rows_here) Q16[row_at(rr) * (DH / 8) + k % (DH / 8)] = bf16x8_to_f16x8_scaled(q[j], scq);
  }
}

// One block per 128-row query tile of one (batch, query head); rows of
// (b, h) are contiguous, n_q of them.
template <int DV, int DH, bool ROPE>
__global__ void __launch_bounds__(256)
attn_bwd_preprocess_kernel(int n_q, int nqt, int Hq, const __grid_constant__ RotaryAngles rot, TensorStrides sq,
                           TensorStrides so, TensorStrides sdo,
                           const uint4* __restrict__ Q, const uint4* __restrict__ O,
                           const uint4* __restrict__ O_lo, const uint4* __restrict__ dO, float* __restrict__ D,
                           float4* __restrict__ tilemax, float4* __restrict__ dQacc, uint4* __restrict__ Q16,
                           uint4* __restrict__ dO16, unsigned int* status) {
  const int64_t bh = blockIdx.x;
  const int qt = blockIdx.y;
  const int64_t i0 = static_cast<int64_t>(qt) * kTileM;
  const int rows_here = static_cast<int>(n_q - i0 < kTileM ? n_q - i0 : kTileM);
  const int64_t row0 = bh * n_q + i0;
  const auto row_at = [row0](int rr) { return row0 + rr; };
  const auto user_at = [bh, i0](const TensorStrides& s, int rr) { return bh * s.head + (i0 + rr) * s.row; };
  const auto tok_at = [bh, Hq, n_q, i0](int rr) { return (bh / Hq) * n_q + i0 + rr; };
  bwd_prep_tile<DV, DH, ROPE>(rows_here, row_at, row_at, user_at, tok_at, rot, sq, so, sdo, Q, O, O_lo, dO, D,
                              tilemax + bh * nqt + qt, dQacc, Q16, dO16, status);
}

// The same for packed sequences (token-major rows, per-sequence lengths):
// row i of (b, h) is token cu_q[b] + i; rows past the sequence's length are
// left alone.
struct PrepPacked {
  int32_t n_q, Hq;
  int64_t total_q;
  TensorStrides sq, so, sdo;
  int32_t cu_q[ATTN_MAX_BATCH + 1];
  __device__ __forceinline__ int64_t len(int b) const { return static_cast<int64_t>(cu_q[b + 1]) - cu_q[b]; }
  __device__ __forceinline__ int64_t row(int b, int h, int64_t i) const {
    return (static_cast<int64_t>(cu_q[b]) + i) * Hq + h;
  }
  __device__ __forceinline__ int64_t vec(int b, int h, int64_t i) const {
    return static_cast<int64_t>(h) * total_q + cu_q[b] + i;
  }
};

template <int DV, int DH, bool ROPE>
__global__ void __launch_bounds__(256)
attn_bwd_preprocess_packed_kernel(const __grid_constant__ PrepPacked rm, int nqt,
                                  const __grid_constant__ RotaryAngles rot, const uint4* __restrict__ Q,
                                  const uint4* __restrict__ O, const uint4* __restrict__ O_lo,
                                  const uint4* __restrict__ dO, float* __restrict__ D, float4* __restrict__ tilemax,
                                  float4* __restrict__ dQacc, uint4* __restrict__ Q16, uint4* __restrict__ dO16,
                                  unsigned int* status) {
  const int64_t bh = blockIdx.x;
  const int b = static_cast<int>(bh / rm.Hq);
  const int h = static_cast<int>(bh - static_cast<int64_t>(b) * rm.Hq);
  const int qt = blockIdx.y;
  const int64_t i0 = static_cast<int64_t>(qt) * kTileM;
  const int64_t left = rm.len(b) - i0;
  const int rows_here = static_cast<int>(left < kTileM ? (left < 0 ? 0 : left) : kTileM);
  const auto row_at = [&rm, b, h, i0](int rr) { return rm.row(b, h, i0 + rr); };
  const auto d_at = [&rm, b, h, i0](int rr) { return rm.vec(b, h, i0 + rr); };
  const int64_t t0 = static_cast<int64_t>(rm.cu_q[b]) + i0;
  const auto user_at = [t0, h](const TensorStrides& s, int rr) { return (t0 + rr) * s.row + h * s.head; };
  const auto tok_at = [t0](int rr) { return t0 + rr; };
  bwd_prep_tile<DV, DH, ROPE>(rows_here, row_at, d_at, user_at, tok_at, rot, rm.sq, rm.so, rm.sdo, Q, O, O_lo, dO, D,
                              tilemax + bh * nqt + qt, dQacc, Q16, dO16, status);
}

// Every query tile of a (batch, KV head) group brought to one exponent for
// its fp16 Q and one for its fp16 dO, the smallest among the group's tiles
// that hold a non-zero entry (f16range.cuh), so that the main kernel's loop
// over the group's steps needs no scale of its own per step.  A tile whose
// own exponent is larger is rescaled in place by the exact power of two
// 2^(e_group - e_tile) < 1: its largest entry lies that many binades below
// the group's largest, and its entries keep full precision down to about
// 2^-28 of the group's largest entry.  The group's exponents go to grpexp
// (0 for a group without any non-zero entry); the tile records are only
// read.  One block per query tile: it reduces its group's records (a few
// hundred bytes from L2) and rescales its own tile if it has to, which
// tiles of similar scale (one exponent, f16range.cuh) never need.
struct GroupExpParams {
  int32_t Hq, Hkv, group, n_q, nqt, packed;
  int32_t cu_q[ATTN_MAX_BATCH + 1];   // packed: first query token of sequence b
  const float4* tilemax;              // [B Hq][nqt]: (.., .., e_Q, e_dO) per tile
  float2* grpexp;                     // [B Hkv]: the group's (e_Q, e_dO)
  uint4* Q16;
  uint4* dO16;
  unsigned int* work_ctr;             // the main kernel's work counter, zeroed here
};

__device__ __forceinline__ uint4 f16x8_scaled(uint4 u, float sc) {
  return make_uint4(pack_f16x2(f16_lo(u.x) * sc, f16_hi(u.x) * sc), pack_f16x2(f16_lo(u.y) * sc, f16_hi(u.y) * sc),
                    pack_f16x2(f16_lo(u.z) * sc, f16_hi(u.z) * sc), pack_f16x2(f16_lo(u.w) * sc, f16_hi(u.w) * sc));
}

// grid (B Hkv, up to group nqt): block (bk, y) takes the tiles idx = y,
// y + gridDim.y, ... of its group, idx naming head hk group + idx / nt and
// query tile idx % nt (nt = the sequence's query tiles).
template <int DH, int DV>
__global__ void __launch_bounds__(256) attn_bwd_group_exp_kernel(const __grid_constant__ GroupExpParams p) {
  const int b = static_cast<int>(blockIdx.x) / p.Hkv;
  const int hk = static_cast<int>(blockIdx.x) - b * p.Hkv;
  const int64_t nq_b = p.packed ? static_cast<int64_t>(p.cu_q[b + 1]) - p.cu_q[b] : p.n_q;
  const int nt = static_cast<int>((nq_b + kTileM - 1) / kTileM);
  const int items = p.group * nt;
  if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) *p.work_ctr = 0u;
  if (static_cast<int>(blockIdx.y) >= items) return;   // past the sequence (packed): no tile
  auto rec_of = [&](int idx) -> const float4* {
    return p.tilemax + static_cast<int64_t>(b * p.Hq + hk * p.group + idx / nt) * p.nqt + idx % nt;
  };
  int qmin = kExpZero, omin = kExpZero;
  for (int idx = static_cast<int>(threadIdx.x); idx < items; idx += 256) {
    const float2 e = reinterpret_cast<const float2*>(rec_of(idx))[1];
    const int q = static_cast<int>(e.x), o = static_cast<int>(e.y);
    if (q != kExpZero) qmin = min(qmin, q);
    if (o != kExpZero) omin = min(omin, o);
  }
  __shared__ int red[2][8];
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    qmin = min(qmin, __shfl_xor_sync(0xffffffffu, qmin, off));
    omin = min(omin, __shfl_xor_sync(0xffffffffu, omin, off));
  }
  if ((threadIdx.x & 31) == 0) {
    red[0][threadIdx.x >> 5] = qmin;
    red[1][threadIdx.x >> 5] = omin;
  }
  __syncthreads();
#pragma unroll
  for (int w = 0; w < 8; ++w) {
    qmin = min(qmin, red[0][w]);
    omin = min(omin, red[1][w]);
  }
  const int qg = qmin == kExpZero ? 0 : qmin, og = omin == kExpZero ? 0 : omin;
  if (blockIdx.y == 0 && threadIdx.x == 0)
    p.grpexp[blockIdx.x] = make_float2(static_cast<float>(qg), static_cast<float>(og));
  for (int self = static_cast<int>(blockIdx.y); self < items; self += static_cast<int>(gridDim.y)) {
  const float2 e = reinterpret_cast<const float2*>(rec_of(self))[1];
  const int q = static_cast<int>(e.x), o = static_cast<int>(e.y);
  const int r = hk * p.group + self / nt;
  const int64_t i0 = static_cast<int64_t>(self % nt) * kTileM;
  const int rows = static_cast<int>(nq_b - i0 < kTileM ? nq_b - i0 : kTileM);
  auto row_at = [&](int rr) -> int64_t {
    return p.packed ? (static_cast<int64_t>(p.cu_q[b]) + i0 + rr) * p.Hq + r
                    : (static_cast<int64_t>(b) * p.Hq + r) * p.n_q + i0 + rr;
  };
  if (q != kExpZero && q != qg) {
    const float sc = exp2_int(qg - q);
    for (int k = static_cast<int>(threadIdx.x); k < rows * (DH / 8); k += 256) {
      uint4* at = p.Q16 + row_at(k / (DH / 8)) * (DH / 8) + k % (DH / 8);
      *at = f16x8_scaled(*at, sc);
    }
  }
  if (o != kExpZero && o != og) {
    const float sc = exp2_int(og - o);
    for (int k = static_cast<int>(threadIdx.x); k < rows * (DV / 8); k += 256) {
      uint4* at = p.dO16 + row_at(k / (DV / 8)) * (DV / 8) + k % (DV / 8);
      *at = f16x8_scaled(*at, sc);
    }
  }
  }
}

// dQ = scale * acc into a strided dQ: the accumulator row r (d_h / 8 chunks of
// 8) is row r % n_inner of group r / n_inner, at element offset
// (r / n_inner) s_outer + (r % n_inner) s_inner (padded: heads of n_q rows;
// packed: tokens of Hq heads).
__global__ void __launch_bounds__(256)
attn_bwd_finalize_strided_kernel(int64_t n8, int c8, int n_inner, int64_t s_outer, int64_t s_inner, float scale,
                                 const float4* __restrict__ acc, uint4* __restrict__ dQ) {
  const int64_t nthreads = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t k = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; k < n8; k += nthreads) {
    const int64_t r = k / c8;
    const int64_t outer = r / n_inner;
    const int64_t off = outer * s_outer + (r - outer * n_inner) * s_inner;
    const float4 a = acc[2 * k];
    const float4 c = acc[2 * k + 1];
    dQ[off / 8 + (k - r * c8)] = make_uint4(pack_bf16x2(a.x * scale, a.y * scale), pack_bf16x2(a.z * scale, a.w * scale),
                                            pack_bf16x2(c.x * scale, c.y * scale), pack_bf16x2(c.z * scale, c.w * scale));
  }
}

// The same with the rotary embedding: each 8-element chunk of the rotated
// query's gradient turned back by its token's angles (the transpose of the
// rotation) before it is rounded.  A work item is one chunk of one token for
// all its query heads, 8 at a time, so that the token's angles are formed
// once per chunk.  Accumulator row and dQ offset of (token, h): padded
// (token = b n_q + i) row (b Hq + h) n_q + i at (b Hq + h) s_head + i s_row;
// packed row token Hq + h at token s_row + h s_head.
__global__ void __launch_bounds__(256)
attn_bwd_finalize_rope_kernel(int64_t tokens, int c8, int Hq, int n_q, int packed, int64_t s_row, int64_t s_head,
                              float scale, const float4* __restrict__ acc, const __grid_constant__ RotaryAngles rot,
                              uint4* __restrict__ dQ) {
  constexpr int kG = 8;
  const int64_t items = tokens * c8;
  const int64_t nthreads = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t u = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; u < items; u += nthreads) {
    const int64_t tok = u / c8;
    const int c = static_cast<int>(u - tok * c8);
    int64_t row0, rstep, off0, ostep;
    if (packed) {
      row0 = tok * Hq;
      rstep = 1;
      off0 = tok * s_row;
      ostep = s_head;
    } else {
      const int64_t b = tok / n_q, i = tok - b * n_q;
      row0 = b * Hq * n_q + i;
      rstep = n_q;
      off0 = b * Hq * s_head + i * s_row;
      ostep = s_head;
    }
    float wh[4], wl[4];
    rope_freqs4(rot.w_hi, rot.w_lo, c, wh, wl);
    float4 t0, t1;
    rope_angles4(rot.pos[tok], wh, wl, t0, t1);
    rope_transpose(t0, t1);
    const float cs[4] = {t0.x, t0.z, t1.x, t1.z}, sn[4] = {t0.y, t0.w, t1.y, t1.w};
    for (int h0 = 0; h0 < Hq; h0 += kG) {
      float4 a[kG], bb[kG];
#pragma unroll
      for (int g = 0; g < kG; ++g)
        if (h0 + g < Hq) {
          const int64_t k = (row0 + (h0 + g) * rstep) * c8 + c;
          a[g] = acc[2 * k];
          bb[g] = acc[2 * k + 1];
        }
#pragma unroll
      for (int g = 0; g < kG; ++g) {
        if (h0 + g >= Hq) break;
        const float x[8] = {a[g].x * scale, a[g].y * scale, a[g].z * scale, a[g].w * scale,
                            bb[g].x * scale, bb[g].y * scale, bb[g].z * scale, bb[g].w * scale};
        uint32_t w[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          float y0, y1;
          rot_block(x[2 * q], x[2 * q + 1], cs[q], sn[q], y0, y1);
          w[q] = pack_bf16x2(y0, y1);
        }
        dQ[(off0 + (h0 + g) * ostep) / 8 + c] = make_uint4(w[0], w[1], w[2], w[3]);
      }
    }
  }
}

// dQ = scale * acc, eight elements per thread per iteration (contiguous dQ).
__global__ void __launch_bounds__(256)
attn_bwd_finalize_kernel(int64_t n8, float scale, const float4* __restrict__ acc, uint4* __restrict__ dQ) {
  const int64_t nthreads = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t k = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; k < n8; k += nthreads) {
    const float4 a = acc[2 * k];
    const float4 c = acc[2 * k + 1];
    dQ[k] = make_uint4(pack_bf16x2(a.x * scale, a.y * scale), pack_bf16x2(a.z * scale, a.w * scale),
                       pack_bf16x2(c.x * scale, c.y * scale), pack_bf16x2(c.z * scale, c.w * scale));
  }
}

__global__ void __launch_bounds__(256) zero_f32_kernel(float4* __restrict__ p, int64_t n4) {
  const int64_t nthreads = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t k = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; k < n4; k += nthreads)
    p[k] = make_float4(0.f, 0.f, 0.f, 0.f);
}

// dK and dV of a query-head split: accumulator row r = token Hkv + h (packed)
// or (b Hkv + h) n_k + j (padded), eight columns per work item, rounded to
// bf16 into the caller's strided tensors.  The K items come first.
struct KvFinParams {
  int64_t rows;                // tokens_k Hkv
  int32_t dh, dv, Hkv, n_k, packed;
  TensorStrides sdk, sdv;
  const float4* dKacc;
  const float4* dVacc;
  uint4* dK;
  uint4* dV;
};

__global__ void __launch_bounds__(256) attn_bwd_kv_finalize_kernel(const __grid_constant__ KvFinParams p) {
  const int64_t items_k = p.rows * (p.dh / 8);
  const int64_t total = items_k + p.rows * (p.dv / 8);
  const int64_t nthreads = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t u0 = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; u0 < total; u0 += nthreads) {
    const bool is_v = u0 >= items_k;
    const int64_t u = is_v ? u0 - items_k : u0;
    const int c8 = (is_v ? p.dv : p.dh) / 8;
    const int64_t r = u / c8;
    const int c = static_cast<int>(u - r * c8);
    int64_t off;
    const TensorStrides& st = is_v ? p.sdv : p.sdk;
    if (p.packed) {
      const int64_t t = r / p.Hkv, h = r - t * p.Hkv;
      off = t * st.row + h * st.head;
    } else {
      const int64_t bh = r / p.n_k, j = r - bh * p.n_k;
      off = bh * st.head + j * st.row;
    }
    const float4* a = (is_v ? p.dVacc : p.dKacc) + u * 2;
    const float4 x = a[0], y = a[1];
    (is_v ? p.dV : p.dK)[off / 8 + c] = make_uint4(pack_bf16x2(x.x, x.y), pack_bf16x2(x.z, x.w),
                                                  pack_bf16x2(y.x, y.y), pack_bf16x2(y.z, y.w));
  }
}

template <int DH, int DV>
cudaError_t launch_bwd_main_t(const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV,
                              const CUtensorMap& tmdO, const CUtensorMap& tmdQ, const BwdParams& p,
                              cudaStream_t stream) {
  using C = BwdCfg<DH, DV>;
  // The split runs without a rotary only (the host never asks for both).
  auto kern = p.rot.pos ? (p.lay.packed ? attn_bwd_main_kernel<DH, DV, true, true, false>
                                        : attn_bwd_main_kernel<DH, DV, false, true, false>)
              : p.hsplit > 1 ? (p.lay.packed ? attn_bwd_main_kernel<DH, DV, true, false, true>
                                             : attn_bwd_main_kernel<DH, DV, false, false, true>)
                             : (p.lay.packed ? attn_bwd_main_kernel<DH, DV, true, false, false>
                                             : attn_bwd_main_kernel<DH, DV, false, false, false>);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (e != cudaSuccess) return e;
  dim3 grid(static_cast<unsigned>(p.sh.B * p.sh.Hkv), static_cast<unsigned>((p.sh.n_k + kTileN - 1) / kTileN),
            static_cast<unsigned>(p.hsplit));
  kern<<<grid, C::kThreads, C::kSmemBytes, stream>>>(tmQ, tmK, tmV, tmdO, tmdQ, p);
  return cudaGetLastError();
}

int grid_for(int64_t work_threads) {
  int64_t blocks = (work_threads + 255) / 256;
  if (blocks < 1) blocks = 1;
  if (blocks > 152 * 64) blocks = 152 * 64;
  return static_cast<int>(blocks);
}

template <int DV, int DH>
void launch_pre_t(const ShapeParams& sh, const LayoutParams& lay, int nqt, const void* Q, const void* O,
                  const void* O_lo, const void* dO, float* D, float4* tilemax, float* dQacc, void* Q16, void* dO16,
                  const RotaryAngles* rot, unsigned int* status, cudaStream_t stream) {
  RotaryAngles none;
  none.pos = nullptr;
  const RotaryAngles& ra = rot ? *rot : none;
  dim3 grid(static_cast<unsigned>(static_cast<int64_t>(sh.B) * sh.Hq), static_cast<unsigned>(nqt));
  const uint4 *q = static_cast<const uint4*>(Q), *o = static_cast<const uint4*>(O);
  const uint4 *olo = static_cast<const uint4*>(O_lo), *g = static_cast<const uint4*>(dO);
  float4* acc = reinterpret_cast<float4*>(dQacc);
  uint4* q16 = static_cast<uint4*>(Q16);
  uint4* do16 = static_cast<uint4*>(dO16);
  if (!lay.packed) {
    auto kern = rot ? attn_bwd_preprocess_kernel<DV, DH, true> : attn_bwd_preprocess_kernel<DV, DH, false>;
    kern<<<grid, 256, 0, stream>>>(sh.n_q, nqt, sh.Hq, ra, lay.sq, lay.so, lay.sdo, q, o, olo, g, D, tilemax, acc,
                                   q16, do16, status);
  } else {
    PrepPacked rm;
    rm.n_q = sh.n_q;
    rm.Hq = sh.Hq;
    rm.total_q = lay.total_q;
    rm.sq = lay.sq;
    rm.so = lay.so;
    rm.sdo = lay.sdo;
    for (int b = 0; b <= sh.B; ++b) rm.cu_q[b] = lay.cu_q[b];
    auto kern = rot ? attn_bwd_preprocess_packed_kernel<DV, DH, true> : attn_bwd_preprocess_packed_kernel<DV, DH, false>;
    kern<<<grid, 256, 0, stream>>>(rm, nqt, ra, q, o, olo, g, D, tilemax, acc, q16, do16, status);
  }
}

}  // namespace

cudaError_t launch_attn_bwd_main(int dh, int dv, const CUtensorMap& tmQ, const CUtensorMap& tmK,
                                 const CUtensorMap& tmV, const CUtensorMap& tmdO, const CUtensorMap& tmdQ,
                                 const BwdParams& p, cudaStream_t stream) {
  if (p.persistent) return launch_attn_bwd_main_persistent(dh, dv, tmQ, tmK, tmV, tmdO, tmdQ, p, stream);
  if (dh == 128 && dv == 128) return launch_bwd_main_t<128, 128>(tmQ, tmK, tmV, tmdO, tmdQ, p, stream);
  if (dh == 64 && dv == 64) return launch_bwd_main_t<64, 64>(tmQ, tmK, tmV, tmdO, tmdQ, p, stream);
  if (dh == 128 && dv == 64) return launch_bwd_main_t<128, 64>(tmQ, tmK, tmV, tmdO, tmdQ, p, stream);
  return cudaErrorInvalidValue;
}

cudaError_t launch_attn_bwd_preprocess(const ShapeParams& sh, const LayoutParams& lay, int dv, int dh,
                                       const void* Q, const void* O, const void* O_lo, const void* dO, float* D,
                                       float4* tilemax, float2* grpexp, unsigned int* work_ctr, float* dQacc,
                                       void* Q16, void* dO16, const RotaryAngles* rot_q, unsigned int* status,
                                       cudaStream_t stream) {
  const int nqt = (sh.n_q + kTileM - 1) / kTileM;
  GroupExpParams g;
  g.Hq = sh.Hq;
  g.Hkv = sh.Hkv;
  g.group = sh.group;
  g.n_q = sh.n_q;
  g.nqt = nqt;
  g.packed = lay.packed;
  for (int b = 0; b <= sh.B; ++b) g.cu_q[b] = lay.packed ? lay.cu_q[b] : 0;
  g.tilemax = tilemax;
  g.grpexp = grpexp;
  g.Q16 = static_cast<uint4*>(Q16);
  g.dO16 = static_cast<uint4*>(dO16);
  g.work_ctr = work_ctr;
  const int64_t gy = static_cast<int64_t>(sh.group) * nqt;
  const dim3 ggrid(static_cast<unsigned>(sh.B * sh.Hkv), static_cast<unsigned>(gy < 65535 ? gy : 65535));
  if (dv == 128 && dh == 128) {
    launch_pre_t<128, 128>(sh, lay, nqt, Q, O, O_lo, dO, D, tilemax, dQacc, Q16, dO16, rot_q, status, stream);
    attn_bwd_group_exp_kernel<128, 128><<<ggrid, 256, 0, stream>>>(g);
  } else if (dv == 64 && dh == 64) {
    launch_pre_t<64, 64>(sh, lay, nqt, Q, O, O_lo, dO, D, tilemax, dQacc, Q16, dO16, rot_q, status, stream);
    attn_bwd_group_exp_kernel<64, 64><<<ggrid, 256, 0, stream>>>(g);
  } else if (dv == 64 && dh == 128) {
    launch_pre_t<64, 128>(sh, lay, nqt, Q, O, O_lo, dO, D, tilemax, dQacc, Q16, dO16, rot_q, status, stream);
    attn_bwd_group_exp_kernel<128, 64><<<ggrid, 256, 0, stream>>>(g);
  } else {
    return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

cudaError_t launch_zero_f32(float* ptr, int64_t n, cudaStream_t stream) {
  const int64_t n4 = n / 4;
  zero_f32_kernel<<<grid_for(n4), 256, 0, stream>>>(reinterpret_cast<float4*>(ptr), n4);
  return cudaGetLastError();
}

cudaError_t launch_attn_bwd_kv_finalize(const ShapeParams& sh, const LayoutParams& lay, int64_t tokens_k, int dh,
                                        int dv, const float* dKacc, const float* dVacc, void* dK, void* dV,
                                        cudaStream_t stream) {
  KvFinParams p;
  p.rows = tokens_k * sh.Hkv;
  p.dh = dh;
  p.dv = dv;
  p.Hkv = sh.Hkv;
  p.n_k = sh.n_k;
  p.packed = lay.packed;
  p.sdk = lay.sdk;
  p.sdv = lay.sdv;
  p.dKacc = reinterpret_cast<const float4*>(dKacc);
  p.dVacc = reinterpret_cast<const float4*>(dVacc);
  p.dK = static_cast<uint4*>(dK);
  p.dV = static_cast<uint4*>(dV);
  attn_bwd_kv_finalize_kernel<<<grid_for(p.rows * ((dh + dv) / 8)), 256, 0, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_attn_bwd_finalize(int64_t elems, int dh, int n_inner, int64_t s_outer, int64_t s_inner,
                                     bool contiguous, float scale, const float* dQacc, void* dQ,
                                     const RotaryAngles* rot_q, bool packed, int Hq, cudaStream_t stream) {
  const int64_t n8 = elems / 8;
  if (rot_q) {
    // Padded rows are heads of n_inner = n_q rows (s_outer the head stride);
    // packed rows are tokens of n_inner = Hq heads (s_outer the token stride).
    const int64_t tokens = elems / (static_cast<int64_t>(Hq) * dh);
    const int64_t items = tokens * (dh / 8);
    attn_bwd_finalize_rope_kernel<<<grid_for(items), 256, 0, stream>>>(
        tokens, dh / 8, Hq, packed ? 0 : n_inner, packed ? 1 : 0, packed ? s_outer : s_inner,
        packed ? s_inner : s_outer, scale, reinterpret_cast<const float4*>(dQacc), *rot_q, static_cast<uint4*>(dQ));
  } else if (contiguous)
    attn_bwd_finalize_kernel<<<grid_for(n8), 256, 0, stream>>>(n8, scale, reinterpret_cast<const float4*>(dQacc),
                                                             static_cast<uint4*>(dQ));
  else
    attn_bwd_finalize_strided_kernel<<<grid_for(n8), 256, 0, stream>>>(
        n8, dh / 8, n_inner, s_outer, s_inner, scale, reinterpret_cast<const float4*>(dQacc), static_cast<uint4*>(dQ));
  return cudaGetLastError();
}

}  // namespace esd
