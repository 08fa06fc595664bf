// attn_fwd.cu -- forward kernel of masked scaled dot-product attention on
// sm_103a: TMA-staged tiles, tcgen05 MMAs into tensor memory, and a
// register-level online softmax.
//
// What it computes ("Appendix A.10 -- Attention matrices and
// backpropagation", eqs. A.10.1-A.10.3): for each query row i,
//   S_ij = scale q_i.k_j on the visible set, A = row softmax with the row
//   maximum subtracted, O = A V, and LSE_i = m_i + ln sum_j exp(S_ij - m_i).
// The blockwise evaluation visits the visible key tiles one at a time and
// keeps a running maximum and running sum per row (the online softmax the
// appendix mentions in section A.10.6); in real arithmetic it is the same
// function, only the rounding order differs.
//
// CTA = two 128-row query tiles of one (batch, query head), sharing every
// K/V tile the CTA loads.  Warp roles (384 threads):
//   warp 0      TMA producer: Q tiles once, then K_j and V_j into rings.
//   warp 1      MMA issuer (converged; one elected lane issues): S_t = Q_t K_j^T
//               into tensor memory, O_t += P_t V_j with P_t read back from
//               tensor memory.
//   warps 2, 3  idle.
//   warps 4-7   softmax for query tile 0 (thread = row = TMEM lane).
//   warps 8-11  softmax for query tile 1.
// V arrives as fp16 from a pre-pass (attn_v16_kernel): every 128-key tile j
// scaled by its own power of two 2^v_j (f16range.cuh), padded key rows
// zeroed.  The softmax writes the weights of tile j as P 2^(E - v_j) with
// one reference E per query tile, so every PV product adds 2^E P V into
// the accumulator and the epilogue divides 2^E out with the row sum.  The
// weights are at most 2^8 (the lazy maximum below), so E may lie up to 7
// above the smallest v_j without overflowing fp16: E = min(vmin + 7, vmax)
// over the tiles the query tile sees, which keeps the weights of tiles with
// up to 2^7 smaller values at full precision.
// While one tile's softmax runs, the tensor core works on the other tile.
//
// Tensor memory (512 columns x 128 lanes x 32 bit):
//   [t*128, t*128+128)   S_t (fp32); P_t (fp16 pairs) overwrites its first
//                        64 columns once the scores are consumed.
//   [256 + t*DV, ...)    O_t accumulator (fp32).
//
// Running-max rescaling is lazy: the reference maximum of a row moves only
// when a new score exceeds it by more than 2^8 in the exp2 domain, so most
// tiles skip the O rescale.  Both the numerator (O) and the denominator (l)
// always use the same reference, so the result is unchanged in real
// arithmetic and no term exceeds 2^8 before normalisation.  The weight of
// the dominant key is then 2^d with d in [0, 8) rather than exactly 1; its
// fp16 rounding leaves at most 2^-11 of relative error in O, which the
// normalisation by the unrounded sum l (the LSE's) keeps (measured: the
// backward's dQ and dK on sharply peaked rows stay within a third of the
// tolerance).  Summing the rounded weights as well would remove it, at three
// more instructions per pair of weights in the hot loop.
//
// The PV product runs in fp16 (weights P and V both re-encoded; V exactly at
// any scale through its tile exponent, P <= 2^8 by the lazy maximum): the
// backward rebuilds the
// weights exactly and takes its row term from this O (c_i = sum_l dO_il O_il,
// eq. A.10.7), so O must be the product of nearly exact weights.  With bf16
// weights (8 significant bits) the two differ by about 2^-9 of
// sum_j P_ij |dP_ij|, which for a sharply peaked row moved dQ past the
// tolerance; fp16 (11 bits) shrinks that eightfold.
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "f16range.cuh"
#include "ptx.cuh"
#include "rotary.cuh"

namespace esd {
namespace {

template <int DH, int DV>
struct FwdCfg {
  static constexpr int kQTiles = 2;
  static constexpr int kKStages = (DH == 128) ? 2 : 3;
  static constexpr int kVStages = 3;
  static constexpr int kQTileBytes = kTileM * DH * 2;
  static constexpr int kKTileBytes = kTileN * DH * 2;
  static constexpr int kVTileBytes = kTileN * DV * 2;
  static constexpr int kBlockBytes = 128 * 128;       // one 128-row x 64-col bf16 block
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kOffQ + kQTiles * kQTileBytes;
  static constexpr int kOffV = kOffK + kKStages * kKTileBytes;
  static constexpr int kOffBar = kOffV + kVStages * kVTileBytes;
  // barrier indices
  static constexpr int kBarQFull = 0;
  static constexpr int kBarKFull = 1;
  static constexpr int kBarKEmpty = kBarKFull + kKStages;
  static constexpr int kBarVFull = kBarKEmpty + kKStages;
  static constexpr int kBarVEmpty = kBarVFull + kVStages;
  static constexpr int kBarSFull = kBarVEmpty + kVStages;    // [2]
  static constexpr int kBarPReady = kBarSFull + 2;          // [2]
  static constexpr int kBarOFull = kBarPReady + 2;          // [2]
  static constexpr int kBarDrain = kBarOFull + 2;
  static constexpr int kNumBars = kBarDrain + 1;
  static constexpr int kOffTmemSlot = kOffBar + kNumBars * 8;
  static constexpr int kOffAbort = kOffTmemSlot + 4;
  static constexpr int kSmemUsed = kOffAbort + 4;
  static constexpr int kSmemBytes = kSmemUsed + 1024;   // slack for 1024-byte alignment
  static constexpr int kThreads = 384;
  static constexpr uint32_t kRegsLaunch = 168;   // 65536 / 384, rounded down to a multiple of 8
  static constexpr uint32_t kRegsLow = 64, kRegsHigh = 216;
  static constexpr uint32_t kTmemCols = 512;
  static_assert(kSmemBytes <= 232448, "shared memory budget");
  static_assert(2 * 128 + 2 * DV <= 512, "tensor memory budget");
};

template <int DH, int DV, bool PACKED>
__global__ void __launch_bounds__(384, 1)
attn_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                const __grid_constant__ CUtensorMap tmV, const __grid_constant__ FwdParams p) {
  using C = FwdCfg<DH, DV>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  auto bar = [&](int idx) -> uint32_t { return sbase + C::kOffBar + 8 * idx; };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffAbort);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffTmemSlot);

  const uint32_t warp = warp_id();
  const uint32_t lane = lane_id();

  // ---- work item ----
  const int bh = blockIdx.x;                        // b * Hq + r
  const int b = bh / p.sh.Hq;
  const int r = bh - b * p.sh.Hq;
  const int hkv = r / p.sh.group;                   // g(r) = r / (Hq / Hkv)
  const int pair = static_cast<int>(gridDim.y) - 1 - static_cast<int>(blockIdx.y);  // heavy first
  int q0[2], ntiles[2];
#pragma unroll
  for (int t = 0; t < 2; ++t) {
    q0[t] = (pair * 2 + t) * kTileM;
    ntiles[t] = kv_tiles_for_q_tile(p.mask, p.sh.n_q, p.sh.n_k, b, q0[t]);
  }
  const int nkv = ntiles[0] > ntiles[1] ? ntiles[0] : ntiles[1];

  // ---- setup ----
  if (threadIdx.x == 0) {
    mbar_init(bar(C::kBarQFull), 1);
    for (int s = 0; s < C::kKStages; ++s) {
      mbar_init(bar(C::kBarKFull + s), 1);
      mbar_init(bar(C::kBarKEmpty + s), 1);
    }
    for (int s = 0; s < C::kVStages; ++s) {
      mbar_init(bar(C::kBarVFull + s), 1);
      mbar_init(bar(C::kBarVEmpty + s), 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(bar(C::kBarSFull + t), 1);
      mbar_init(bar(C::kBarPReady + t), 128);
      mbar_init(bar(C::kBarOFull + t), 1);
    }
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
  // Registers: the producer/MMA warpgroup gives up most of its share to the
  // two softmax warpgroups, which hold a whole 128-column score row each
  // (128 x 56 + 256 x 224 = 384 x 168, the launch allocation).
  static_assert(128 * C::kRegsLow + 256 * C::kRegsHigh <= C::kThreads * C::kRegsLaunch, "register split");

  if (warp < 4) setmaxnreg_to<C::kRegsLow, C::kRegsLaunch>();
  if (warp == 0) {
    // =========================== TMA producer ===========================
    if (lane == 0 && *abort_flag == 0) {
      tma_prefetch_map(&tmQ);
      tma_prefetch_map(&tmK);
      tma_prefetch_map(&tmV);
      TmaYZ qyz[2];
      for (int t = 0; t < C::kQTiles; ++t) qyz[t] = q_tma(PACKED, p.lay, p.sh.Hq, b, r, q0[t]);
      mbar_arrive_expect_tx(bar(C::kBarQFull), C::kQTiles * C::kQTileBytes);
      for (int t = 0; t < C::kQTiles; ++t)
        for (int c = 0; c < DH / 64; ++c)
          tma_load_3d(sbase + C::kOffQ + t * C::kQTileBytes + c * C::kBlockBytes, &tmQ,
                      bar(C::kBarQFull), c * 64, qyz[t].y, qyz[t].z);
      int k_issued[C::kKStages > C::kVStages ? C::kKStages : C::kVStages] = {};
      int v_issued[C::kKStages > C::kVStages ? C::kKStages : C::kVStages] = {};
      bool ok = true;
      for (int j = 0; j < nkv && ok; ++j) {
        const int ks = j % C::kKStages;
        const uint32_t kph = static_cast<uint32_t>((j / C::kKStages) & 1);
        ok = mbar_wait(bar(C::kBarKEmpty + ks), kph ^ 1u, abort_flag, limit);
        if (!ok) break;
        mbar_arrive_expect_tx(bar(C::kBarKFull + ks), C::kKTileBytes);
        const TmaYZ kyz = k_tma(PACKED, p.lay, p.sh.Hkv, b, hkv, j * kTileN);
        for (int c = 0; c < DH / 64; ++c)
          tma_load_3d(sbase + C::kOffK + ks * C::kKTileBytes + c * C::kBlockBytes, &tmK,
                      bar(C::kBarKFull + ks), c * 64, kyz.y, kyz.z);
        ++k_issued[ks];
        const int vs = j % C::kVStages;
        const uint32_t vph = static_cast<uint32_t>((j / C::kVStages) & 1);
        ok = mbar_wait(bar(C::kBarVEmpty + vs), vph ^ 1u, abort_flag, limit);
        if (!ok) break;
        mbar_arrive_expect_tx(bar(C::kBarVFull + vs), C::kVTileBytes);
        // V16 is [B Hkv][nkt 128][DV] in both layouts.
        for (int c = 0; c < DV / 64; ++c)
          tma_load_3d(sbase + C::kOffV + vs * C::kVTileBytes + c * C::kBlockBytes, &tmV,
                      bar(C::kBarVFull + vs), c * 64, j * kTileN, b * p.sh.Hkv + hkv);
        ++v_issued[vs];
      }
      if (*abort_flag) {
        // Let every copy already in flight land before the CTA can exit.
        int no_abort = 0;
        mbar_wait(bar(C::kBarQFull), 0, &no_abort, limit);
        for (int s = 0; s < C::kKStages; ++s)
          if (k_issued[s]) mbar_wait(bar(C::kBarKFull + s), (k_issued[s] - 1) & 1, &no_abort, limit);
        for (int s = 0; s < C::kVStages; ++s)
          if (v_issued[s]) mbar_wait(bar(C::kBarVFull + s), (v_issued[s] - 1) & 1, &no_abort, limit);
      }
    }
  } else if (warp == 1) {
    // ============================ MMA issuer ============================
    // The whole warp follows the schedule and one elected lane issues: the
    // descriptors and tensor-memory addresses stay warp-uniform, which keeps
    // the issue rate while the softmax warps sharing this sub-partition take
    // most issue slots.  Waits end in a vote, so the warp stays converged.
    if (__all_sync(0xffffffffu, *abort_flag == 0)) {
      constexpr uint32_t kIdescQK = idesc_bf16_f32(128, 128, false, false);
      constexpr uint32_t kIdescPV = idesc_f16_f32(128, DV, false, true);   // fp16 P and V
      // Shared-memory descriptors as base words plus constant steps: every
      // instruction between two MMAs delays the tensor core.
      const SmemDesc dq0 = sw128_desc_words(sbase + C::kOffQ, 16, 1024);
      const SmemDesc dk0 = sw128_desc_words(sbase + C::kOffK, 16, 1024);
      const SmemDesc dv0 = sw128_desc_words(sbase + C::kOffV, C::kBlockBytes, 1024);
      auto issue_qk = [&](int t, int ks) {   // S_t = Q_t K^T
        const SmemDesc dq = desc_step(dq0, t * C::kQTileBytes);
        const SmemDesc dk = desc_step(dk0, ks * C::kKTileBytes);
#pragma unroll
        for (int kk = 0; kk < DH / 16; ++kk) {
          const uint32_t off = (kk >> 2) * C::kBlockBytes + (kk & 3) * 32;
          umma_ss_we(tmem + t * 128, desc_step(dq, off), desc_step(dk, off), kIdescQK, kk > 0 ? 1u : 0u);
        }
      };
      auto issue_pv = [&](int t, int vs, bool accumulate) {   // O_t += P_t V
        const SmemDesc dv = desc_step(dv0, vs * C::kVTileBytes);
#pragma unroll
        for (int kk = 0; kk < kTileN / 16; ++kk)
          umma_ts_we(tmem + 256 + t * DV, tmem + t * 128 + kk * 8, desc_step(dv, kk * 16 * 128), kIdescPV,
                    (accumulate || kk > 0) ? 1u : 0u);
      };
      auto wait1 = [&](int idx, uint32_t parity) -> bool {
        return __all_sync(0xffffffffu, mbar_wait(bar(idx), parity, abort_flag, limit));
      };
      bool ok = wait1(C::kBarQFull, 0);
      if (ok && nkv > 0) {
        ok = wait1(C::kBarKFull + 0, 0);
        if (ok) {
          tc_fence_after_sync();
          for (int t = 0; t < 2; ++t)
            if (ntiles[t] > 0) {
              issue_qk(t, 0);
              umma_commit_we(bar(C::kBarSFull + t));
            }
          umma_commit_we(bar(C::kBarKEmpty + 0));
        }
      }
      for (int j = 0; j < nkv && ok; ++j) {
        const int vs = j % C::kVStages;
        ok = wait1(C::kBarVFull + vs, static_cast<uint32_t>((j / C::kVStages) & 1));
        if (!ok) break;
        const int kn = (j + 1) % C::kKStages;
        bool k_next_ready = false;
        for (int t = 0; t < 2 && ok; ++t) {
          if (j < ntiles[t]) {
            ok = wait1(C::kBarPReady + t, static_cast<uint32_t>(j & 1));
            if (!ok) break;
            tc_fence_after_sync();
            issue_pv(t, vs, j > 0);
            if (j == ntiles[t] - 1) umma_commit_we(bar(C::kBarOFull + t));
          }
          if (j + 1 < ntiles[t]) {
            if (!k_next_ready) {
              ok = wait1(C::kBarKFull + kn, static_cast<uint32_t>(((j + 1) / C::kKStages) & 1));
              if (!ok) break;
              tc_fence_after_sync();
              k_next_ready = true;
            }
            issue_qk(t, kn);
            umma_commit_we(bar(C::kBarSFull + t));
          }
        }
        if (!ok) break;
        umma_commit_we(bar(C::kBarVEmpty + vs));
        if (k_next_ready) umma_commit_we(bar(C::kBarKEmpty + kn));
      }
      // Every MMA issued above must finish before tensor memory is freed.
      int no_abort = 0;
      umma_commit_we(bar(C::kBarDrain));
      mbar_wait(bar(C::kBarDrain), 0, &no_abort, limit);
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ============================== softmax =============================
    setmaxnreg_to<C::kRegsHigh, C::kRegsLaunch>();
    const int t = (warp - 4) / 4;
    const uint32_t quad = warp & 3;
    const int row = static_cast<int>(quad * 32 + lane);
    const int64_t i = static_cast<int64_t>(q0[t]) + row;
    const int64_t lim = row_key_limit(p.mask, p.sh.n_k, b, i);
    const uint32_t lane_base = (quad * 32u) << 16;
    const uint32_t tS = tmem + lane_base + t * 128;
    const uint32_t tO = tmem + lane_base + 256 + t * DV;
    const float sl2 = p.scale_log2;
    float m_ref = -INFINITY;   // reference maximum, exp2 domain
    float l_sum = 0.f;         // sum of the weights p
    bool ok = *abort_flag == 0;
    uint32_t rr[32];
    // The reference E of this query tile's V exponents (all-zero tiles left
    // out), and each tile's offset E - v_j <= 7 for its weights.
    const int* vexp = p.vexp + static_cast<int64_t>(b * p.sh.Hkv + hkv) * p.nkt;
    int vmin = kExpZero, vmax = -kExpZero;
    for (int jt = static_cast<int>(lane); jt < ntiles[t]; jt += 32) {
      const int e = vexp[jt];
      if (e != kExpZero) {
        vmin = min(vmin, e);
        vmax = max(vmax, e);
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      vmin = min(vmin, __shfl_xor_sync(0xffffffffu, vmin, off));
      vmax = max(vmax, __shfl_xor_sync(0xffffffffu, vmax, off));
    }
    const int vref = vmin == kExpZero ? 0 : min(vmin + 7, vmax);
    int v_next = ntiles[t] > 0 ? vexp[0] : 0;
    for (int j = 0; j < ntiles[t] && ok; ++j) {
      const int v_j = v_next;
      if (j + 1 < ntiles[t]) v_next = vexp[j + 1];
      const int voff = v_j == kExpZero ? 0 : vref - v_j;
      ok = __all_sync(0xffffffffu,
                      mbar_wait(bar(C::kBarSFull + t), static_cast<uint32_t>(j & 1), abort_flag, limit));
      if (!ok) break;
      tc_fence_after_sync();
      int64_t lrel64 = lim - static_cast<int64_t>(j) * kTileN;
      const int lim_rel = lrel64 > kTileN ? kTileN : (lrel64 < 0 ? 0 : static_cast<int>(lrel64));
      const bool masked = __any_sync(0xffffffffu, lim_rel < kTileN);

      // The whole 128-column score row in registers: four loads, one wait.
      uint32_t sc[4][32];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld32_nowait(tS + c * 32, sc[c]);
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_wait_ld32(sc[c]);
      // Scores outside the visible set become -inf, so their weights below
      // are exp2(-inf) = 0 without a second test.
      if (masked) {
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int k = 0; k < 32; ++k)
            sc[c][k] = (c * 32 + k < lim_rel) ? sc[c][k] : __float_as_uint(-INFINITY);
      }
      // Row maximum: four independent chains of three-input maxima.
      float mxc[4];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        mxc[c] = fmaxf(__uint_as_float(sc[c][0]), __uint_as_float(sc[c][1]));
#pragma unroll
        for (int k = 2; k < 32; k += 2) mxc[c] = fmax3(mxc[c], __uint_as_float(sc[c][k]), __uint_as_float(sc[c][k + 1]));
      }
      const float mx = fmaxf(fmaxf(mxc[0], mxc[1]), fmaxf(mxc[2], mxc[3]));
      const float m_new = fmaxf(m_ref, mx * sl2);
      if (j == 0) {
        m_ref = m_new;
      } else {
        const bool need = m_new > m_ref + 8.0f;
        if (__any_sync(0xffffffffu, need)) {
          const float alpha = need ? fast_exp2(m_ref - m_new) : 1.0f;
          if (need) {
            l_sum *= alpha;
            m_ref = m_new;
          }
#pragma unroll
          for (int c = 0; c < DV / 32; ++c) {
            tmem_ld32(tO + c * 32, rr);
#pragma unroll
            for (int k = 0; k < 32; ++k) rr[k] = __float_as_uint(__uint_as_float(rr[k]) * alpha);
            tmem_st32(tO + c * 32, rr);
          }
        }
      }
      const float nm = ((m_ref == -INFINITY) ? 0.f : -m_ref) + static_cast<float>(voff);

      // P' = exp2(S scale log2e - m_ref + E - v_j) -> fp16 pairs into
      // tensor memory (over the first 64 columns of S, all of which are in
      // registers); the row sum takes P = P' 2^(v_j - vmin).
      float ls[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t pw[16];
#pragma unroll
        for (int k = 0; k < 32; k += 2) {
          float x0, x1;
          ffma2(x0, x1, __uint_as_float(sc[c][k]), __uint_as_float(sc[c][k + 1]), sl2, sl2, nm, nm);
          const float p0 = fast_exp2(x0), p1 = fast_exp2(x1);
          const uint32_t w = pack_f16x2(p0, p1);
          fadd2(ls[c & 1][0], ls[c & 1][1], p0, p1);
          pw[k >> 1] = w;
        }
        tmem_st16_nowait(tS + c * 16, pw);
      }
      l_sum += ((ls[0][0] + ls[0][1]) + (ls[1][0] + ls[1][1])) * exp2_int(-voff);
      tmem_wait_st();
      tc_fence_before_sync();
      mbar_arrive(bar(C::kBarPReady + t));
    }

    // ---- epilogue: O = acc / l, LSE = (m_ref + log2 l) ln 2 ----
    if (ok && ntiles[t] > 0) {
      ok = __all_sync(0xffffffffu, mbar_wait(bar(C::kBarOFull + t), 0, abort_flag, limit));
      tc_fence_after_sync();
      if (ok) {
        // O = 2^-E acc / l (the weights of tile j were scaled by 2^(E - v_j)).
        const float inv_l = l_sum > 0.f ? exp2_int(-vref) / l_sum : 0.f;
        const bool in_range = i < query_len(p.mask, p.sh.n_q, b);
        const int64_t row_off = strided_off(PACKED, p.lay.so, p.sh.Hq, p.lay.cu_q[b], b, r, i);
        uint4* orow = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.O) + row_off);
        uint4* lorow = p.O_lo ? reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.O_lo) + row_off) : nullptr;
#pragma unroll
        for (int c = 0; c < DV / 32; ++c) {
          tmem_ld32(tO + c * 32, rr);
          uint32_t w[16], lo[16];
#pragma unroll
          for (int k = 0; k < 32; k += 2) {
            const float o0 = __uint_as_float(rr[k]) * inv_l, o1 = __uint_as_float(rr[k + 1]) * inv_l;
            w[k >> 1] = pack_bf16x2(o0, o1);
            lo[k >> 1] = pack_bf16x2(o0 - bf16_lo(w[k >> 1]), o1 - bf16_hi(w[k >> 1]));
          }
          if (in_range) {
#pragma unroll
            for (int v = 0; v < 4; ++v)
              orow[c * 4 + v] = make_uint4(w[4 * v], w[4 * v + 1], w[4 * v + 2], w[4 * v + 3]);
            if (lorow) {
#pragma unroll
              for (int v = 0; v < 4; ++v)
                lorow[c * 4 + v] = make_uint4(lo[4 * v], lo[4 * v + 1], lo[4 * v + 2], lo[4 * v + 3]);
            }
          }
        }
        if (in_range)
          p.LSE[q_vec(PACKED, p.lay, p.sh.Hq, p.sh.n_q, b, r, i)] = (m_ref + fast_log2(l_sum)) * kLn2;
      }
    }
  }

  // ---- teardown ----
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, C::kTmemCols);
  }
  if (threadIdx.x == 0 && *abort_flag == 1) record_status(p.status, ATTN_ERR_TIMEOUT);
}

// V for the forward's P V product: every 128-key tile of (b, h) re-encoded
// as fp16 x 2^e, e from the tile's largest magnitude (f16range.cuh), rows
// past the key length zero, and e recorded in vexp.  One block per tile;
// the whole tile stays in registers while the block agrees on e.  Tiles that
// start past the key length are never read by the forward and are skipped.
template <int DV, bool PACKED, bool ROPE>
__global__ void __launch_bounds__(256) attn_v16_kernel(const __grid_constant__ V16Params p) {
  constexpr int kCpr = DV / 8;                    // 16-byte chunks per row
  constexpr int kChunks = kTileN * kCpr / 256;    // per thread
  if (ROPE && static_cast<int>(blockIdx.y) >= p.nkt) {
    // Rotary: the rotated queries and keys, in the same launch.
    const int64_t blk = static_cast<int64_t>(blockIdx.y - p.nkt) * gridDim.x + blockIdx.x;
    rope_prep_range(p.rp, blk * 256 + threadIdx.x, static_cast<int64_t>(p.prep_rows) * gridDim.x * 256);
    return;
  }
  const int bh = blockIdx.x;
  const int b = bh / p.sh.Hkv;
  const int h = bh - b * p.sh.Hkv;
  const int64_t j0 = static_cast<int64_t>(blockIdx.y) * kTileN;
  const int64_t klen = key_len(p.mask, p.sh.n_k, b);
  if (j0 >= klen) return;
  __shared__ float red[8];
  const uint4* V = static_cast<const uint4*>(p.V);
  uint4 v[kChunks];
  uint32_t m = 0u;
#pragma unroll
  for (int i = 0; i < kChunks; ++i) {
    const int k = static_cast<int>(threadIdx.x) + 256 * i;
    const int64_t jr = j0 + k / kCpr;
    v[i] = make_uint4(0u, 0u, 0u, 0u);
    if (jr < klen) {
      v[i] = V[strided_off(PACKED, p.lay.sv, p.sh.Hkv, p.lay.cu_k[b], b, h, jr) / 8 + k % kCpr];
      m = bf16_absmax_fold(m, v[i]);
    }
  }
  float mx = bf16_absmax_value(m);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = mx;
  __syncthreads();
#pragma unroll
  for (int w = 0; w < 8; ++w) mx = fmaxf(mx, red[w]);
  const int e = f16_tile_exponent(mx);
  const float sc = exp2_int(e == kExpZero ? 0 : e);
  uint4* dst = static_cast<uint4*>(p.V16) + (static_cast<int64_t>(bh) * p.nkt * kTileN + j0) * kCpr;
#pragma unroll
  for (int i = 0; i < kChunks; ++i) {
    const int k = static_cast<int>(threadIdx.x) + 256 * i;
    dst[k] = (j0 + k / kCpr < klen) ? bf16x8_to_f16x8_scaled(v[i], sc) : make_uint4(0u, 0u, 0u, 0u);
  }
  if (threadIdx.x == 0) {
    p.vexp[static_cast<int64_t>(bh) * p.nkt + blockIdx.y] = e;
    if (f16_saturates(mx, e)) record_status(p.status, ATTN_ERR_RANGE);
  }
}

template <int DH, int DV>
cudaError_t launch_fwd_t(const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV,
                         const FwdParams& p, cudaStream_t stream) {
  using C = FwdCfg<DH, DV>;
  auto kern = p.lay.packed ? attn_fwd_kernel<DH, DV, true> : attn_fwd_kernel<DH, DV, false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (e != cudaSuccess) return e;
  const int pairs = (p.sh.n_q + 2 * kTileM - 1) / (2 * kTileM);
  dim3 grid(static_cast<unsigned>(p.sh.B * p.sh.Hq), static_cast<unsigned>(pairs));
  kern<<<grid, C::kThreads, C::kSmemBytes, stream>>>(tmQ, tmK, tmV, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attn_v16(int dv, const V16Params& p, cudaStream_t stream) {
  const dim3 grid(static_cast<unsigned>(p.sh.B * p.sh.Hkv), static_cast<unsigned>(p.nkt + p.prep_rows));
  const bool rope = p.prep_rows > 0;
  decltype(&attn_v16_kernel<128, true, true>) kern;
  if (dv == 128)
    kern = p.lay.packed ? (rope ? attn_v16_kernel<128, true, true> : attn_v16_kernel<128, true, false>)
                        : (rope ? attn_v16_kernel<128, false, true> : attn_v16_kernel<128, false, false>);
  else if (dv == 64)
    kern = p.lay.packed ? (rope ? attn_v16_kernel<64, true, true> : attn_v16_kernel<64, true, false>)
                        : (rope ? attn_v16_kernel<64, false, true> : attn_v16_kernel<64, false, false>);
  else
    return cudaErrorInvalidValue;
  kern<<<grid, 256, 0, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_attn_fwd(int dh, int dv, const CUtensorMap& tmQ, const CUtensorMap& tmK,
                            const CUtensorMap& tmV, const FwdParams& p, cudaStream_t stream) {
  if (dh == 128 && dv == 128) return launch_fwd_t<128, 128>(tmQ, tmK, tmV, p, stream);
  if (dh == 64 && dv == 64) return launch_fwd_t<64, 64>(tmQ, tmK, tmV, p, stream);
  if (dh == 128 && dv == 64) return launch_fwd_t<128, 64>(tmQ, tmK, tmV, p, stream);
  return cudaErrorInvalidValue;
}

}  // namespace esd
