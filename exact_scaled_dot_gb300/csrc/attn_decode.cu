// attn_decode.cu -- forward attention for short query blocks over a long key
// cache (decode, small chunks of new queries), on sm_103a.
//
// Same function as the forward kernel ("Appendix A.10 -- Attention matrices
// and backpropagation", eqs. A.10.1-A.10.3; the new-queries-over-a-history
// shape of "Chapter 31 -- attention backprop", section 1): O = softmax(S) V
// and the log-sum-exp per query row, over the same visible sets.  What
// differs is how the work is laid out:
//
// * Row packing.  With n_q <= 128 a query head fills only n_q rows of a
//   128-row tile, so the query heads that share a KV head are packed into
//   one tile: row r holds query (r mod n_q) of head (r div n_q) of the
//   chunk.  Every K/V tile is then streamed once for the whole group.  The
//   rows are gathered by threads (no per-head padding to the TMA box).
// * Split key range.  The visible key tiles of a row tile are divided into
//   `nsplit` contiguous ranges processed by different CTAs, so that a few
//   row tiles still fill the GPU.  Each range yields a partial output
//   normalised within the range and its log-sum-exp; the merge kernel
//   combines them, O = sum_s exp(LSE_s - LSE) O_s with LSE = log sum_s
//   exp(LSE_s), which is the same softmax in real arithmetic.
// * One row tile per CTA; the scores run one key tile ahead of the softmax
//   in two buffers: QK(j+1) is computed while the softmax works on tile j,
//   and QK(j+2) is issued right behind PV(j), which has read P(j) out of the
//   buffer QK(j+2) overwrites (the tensor core runs one thread's products
//   in order).  A softmax warp can then be one tile ahead of the others,
//   which is why the P-ready barriers are per buffer, and a warp that has
//   finished its last tile may find two PV products still pending, which is
//   why the last one completes a barrier of its own (a parity wait on the
//   PV-done barrier would match the phase before them).
//
// CTA: 256 threads.  warp 0 TMA producer (K and V tiles, three-stage
// rings), warp 1 MMA issuer (converged, one elected lane issues), warp 2
// gathers Q and then zeroes padded V rows as tiles land, warp 3 helps gather
// Q, warps 4-7 softmax (thread = row).
// Tensor memory: scores of even and odd key tiles in S_0 [0,128) and
// S_1 [128,256) (P as bf16 pairs over the first 64 columns of its buffer),
// O [256, 256 + DV).
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "f16range.cuh"
#include "ptx.cuh"

namespace esd {
namespace {

template <int DH, int DV>
struct DecCfg {
  static constexpr int kBoxBytes = 128 * 128;
  static constexpr int kQTileBytes = 128 * DH * 2;
  static constexpr int kKTileBytes = 128 * DH * 2;
  static constexpr int kVTileBytes = 128 * DV * 2;
  // K and V rings of three stages: a CTA streams its key range once, so
  // the more tiles in flight, the more of the HBM latency is hidden.
  static constexpr int kStages = 3;
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kOffQ + kQTileBytes;
  static constexpr int kOffV = kOffK + kStages * kKTileBytes;
  static constexpr int kOffBar = kOffV + kStages * kVTileBytes;
  static constexpr int kBarQReady = 0;
  static constexpr int kBarKFull = 1;                        // [kStages]
  static constexpr int kBarKEmpty = kBarKFull + kStages;     // [kStages]
  static constexpr int kBarVFull = kBarKEmpty + kStages;     // [kStages]
  static constexpr int kBarVReady = kBarVFull + kStages;     // [kStages]
  static constexpr int kBarVEmpty = kBarVReady + kStages;    // [kStages]
  static constexpr int kBarSFull = kBarVEmpty + kStages;     // [2], one per score buffer
  // [2], one per score buffer: a softmax warp may run one tile ahead of the
  // others (the scores of tile j+1 are computed before P(j) is complete), so
  // its arrival for tile j+1 must not count towards tile j.
  static constexpr int kBarPReady = kBarSFull + 2;
  static constexpr int kBarPVDone = kBarPReady + 2;
  static constexpr int kBarOFull = kBarPVDone + 1;     // the last PV product done (single use)
  static constexpr int kBarDrain = kBarOFull + 1;
  static constexpr int kNumBars = kBarDrain + 1;
  static constexpr int kOffTmemSlot = kOffBar + kNumBars * 8;
  static constexpr int kOffAbort = kOffTmemSlot + 4;
  static constexpr int kSmemUsed = kOffAbort + 4;
  static constexpr int kSmemBytes = kSmemUsed + 1024;   // slack for 1024-byte alignment
  static constexpr int kThreads = 256;
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kTO = 256;
  static_assert(kSmemBytes <= 232448, "shared memory budget");
  static_assert(kTO + DV <= kTmemCols, "tensor memory budget");
};

template <int DH, int DV>
__global__ void __launch_bounds__(256, 1)
attn_decode_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                   const __grid_constant__ DecParams p) {
  using C = DecCfg<DH, DV>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  auto bar = [&](int idx) -> uint32_t { return sbase + C::kOffBar + 8 * idx; };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffAbort);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffTmemSlot);

  const uint32_t warp = warp_id();
  const uint32_t lane = lane_id();

  // ---- work item: row tile (batch, KV head, head chunk) and key range ----
  // Row tiles run fastest in the dispatch order, batch by batch in
  // batch_order (the longest key range first), so that the last CTAs to
  // start are the short batches' last key ranges.
  const int chunks = p.chunks;
  const int tile = blockIdx.x;
  const int rkv = tile / chunks;                      // rank * Hkv + hkv
  const int chunk = tile - rkv * chunks;
  const int b_rank = rkv / p.sh.Hkv;
  const int hkv = rkv - b_rank * p.sh.Hkv;
  const int b = p.batch_order[b_rank];
  const int bkv = b * p.sh.Hkv + hkv;
  const int split = blockIdx.y;
  const int n_q = p.sh.n_q;
  // Rows r < rows_valid hold (head h0 + r / n_q, query r % n_q).
  const int h0 = chunk * p.heads_per_tile;
  int heads_here = p.sh.group - h0;
  if (heads_here > p.heads_per_tile) heads_here = p.heads_per_tile;
  const int rows_valid = heads_here * n_q;
  // Key tiles of the longest row (the last query), split into ranges.
  const int64_t lim_max = row_key_limit(p.mask, p.sh.n_k, b, static_cast<int64_t>(n_q) - 1);
  const int ntiles = lim_max > 0 ? static_cast<int>((lim_max + kTileN - 1) / kTileN) : 0;
  const int t0 = static_cast<int>((static_cast<int64_t>(ntiles) * split) / p.nsplit);
  const int t1 = static_cast<int>((static_cast<int64_t>(ntiles) * (split + 1)) / p.nsplit);
  const int n = t1 - t0;

  // ---- setup ----
  if (threadIdx.x == 0) {
    mbar_init(bar(C::kBarQReady), 64);
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(bar(C::kBarKFull + s), 1);
      mbar_init(bar(C::kBarKEmpty + s), 1);
      mbar_init(bar(C::kBarVFull + s), 1);
      mbar_init(bar(C::kBarVReady + s), 1);
      mbar_init(bar(C::kBarVEmpty + s), 1);
    }
    for (int s = 0; s < 2; ++s) mbar_init(bar(C::kBarSFull + s), 1);
    mbar_init(bar(C::kBarPReady + 0), 128);
    mbar_init(bar(C::kBarPReady + 1), 128);
    mbar_init(bar(C::kBarPVDone), 1);
    mbar_init(bar(C::kBarOFull), 1);
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
  const int64_t klen = key_len(p.mask, p.sh.n_k, b);

  if (warp == 0) {
    // ====================== TMA producer: K and V tiles ==================
    if (lane == 0 && *abort_flag == 0 && n > 0) {
      tma_prefetch_map(&tmK);
      tma_prefetch_map(&tmV);
      int k_issued[C::kStages] = {}, v_issued[C::kStages] = {};
      for (int j = 0; j < n; ++j) {
        const int st = j % C::kStages;
        const uint32_t ph = static_cast<uint32_t>((j / C::kStages - 1) & 1);
        const int32_t row = (t0 + j) * kTileN;
        if (j >= C::kStages && !mbar_wait(bar(C::kBarKEmpty + st), ph, abort_flag, limit)) break;
        mbar_arrive_expect_tx(bar(C::kBarKFull + st), C::kKTileBytes);
        for (int c = 0; c < DH / 64; ++c)
          tma_load_3d(sbase + C::kOffK + st * C::kKTileBytes + c * C::kBoxBytes, &tmK, bar(C::kBarKFull + st),
                      c * 64, row, bkv);
        ++k_issued[st];
        if (j >= C::kStages && !mbar_wait(bar(C::kBarVEmpty + st), ph, abort_flag, limit)) break;
        mbar_arrive_expect_tx(bar(C::kBarVFull + st), C::kVTileBytes);
        for (int c = 0; c < DV / 64; ++c)
          tma_load_3d(sbase + C::kOffV + st * C::kVTileBytes + c * C::kBoxBytes, &tmV, bar(C::kBarVFull + st),
                      c * 64, row, bkv);
        ++v_issued[st];
      }
      if (*abort_flag) {
        int no_abort = 0;
        for (int s = 0; s < C::kStages; ++s) {
          if (k_issued[s]) mbar_wait(bar(C::kBarKFull + s), (k_issued[s] - 1) & 1, &no_abort, limit);
          if (v_issued[s]) mbar_wait(bar(C::kBarVFull + s), (v_issued[s] - 1) & 1, &no_abort, limit);
        }
      }
    }
  } else if (warp == 2 || warp == 3) {
    // ==== gather Q rows into the swizzled tile; then padded V rows =======
    // Row r of the tile is query i = r % n_q of query head h0 + r / n_q;
    // rows past rows_valid are zeros.  Layout: 64-column blocks of 128 rows
    // x 128 bytes, the 16-byte chunk index XOR-swizzled with the row, as the
    // MMA's K-major operand descriptor expects.
    const int t = static_cast<int>(threadIdx.x) - 64;   // 0..63
    const __nv_bfloat16* Q = static_cast<const __nv_bfloat16*>(p.Q);
    const int bh_base = b * p.sh.Hq + hkv * p.sh.group + h0;
    if (*abort_flag == 0 && n > 0) {
      for (int c = t; c < 128 * (DH / 8); c += 64) {
        const int r = c / (DH / 8);
        const int k = c - r * (DH / 8);            // 16-byte chunk of the row
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (r < rows_valid) {
          const int hh = r / n_q, i = r - hh * n_q;
          v = *reinterpret_cast<const uint4*>(Q + ((static_cast<int64_t>(bh_base + hh) * n_q + i) * DH + k * 8));
        }
        *reinterpret_cast<uint4*>(smem + C::kOffQ + (k / 8) * C::kBoxBytes + r * 128 + (((k % 8) ^ (r & 7)) * 16)) =
            v;
      }
      fence_proxy_async_smem();
    }
    mbar_arrive(bar(C::kBarQReady));
    if (warp == 2) {
      // Key rows in [kv_len, n_k) hold caller memory that may be anything
      // (even NaN); their weights are exactly 0, but 0 * NaN would still
      // poison O, so those V rows are zeroed before the PV product.
      bool ok = *abort_flag == 0;
      for (int j = 0; j < n && ok; ++j) {
        const int st = j % C::kStages;
        ok = __all_sync(0xffffffffu, mbar_wait(bar(C::kBarVFull + st), static_cast<uint32_t>((j / C::kStages) & 1),
                                               abort_flag, limit));
        if (!ok) break;
        const int64_t base = static_cast<int64_t>(t0 + j) * kTileN;
        int64_t r0 = klen - base, r1 = static_cast<int64_t>(p.sh.n_k) - base;
        if (r0 < 0) r0 = 0;
        if (r1 > kTileN) r1 = kTileN;
        if (r0 < r1) {
          uint8_t* vbase = smem + C::kOffV + st * C::kVTileBytes;
          const int nch = static_cast<int>(r1 - r0) * (DV / 64) * 8;
          for (int q = static_cast<int>(lane); q < nch; q += 32) {
            const int row = static_cast<int>(r0) + q / ((DV / 64) * 8);
            const int rem = q % ((DV / 64) * 8);
            *reinterpret_cast<uint4*>(vbase + (rem / 8) * C::kBoxBytes + row * 128 + (rem % 8) * 16) =
                make_uint4(0u, 0u, 0u, 0u);
          }
          fence_proxy_async_smem();
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(C::kBarVReady + st));
      }
    }
  } else if (warp == 1) {
    // ============================ MMA issuer ============================
    // The whole warp follows the schedule (waits end in a vote) and one
    // elected lane issues, so that descriptors stay warp-uniform.
    if (__all_sync(0xffffffffu, *abort_flag == 0) && n > 0) {
      constexpr uint32_t kIdQK = idesc_bf16_f32(128, 128, false, false);
      constexpr uint32_t kIdPV = idesc_bf16_f32(128, DV, false, true);
      auto wait1 = [&](int idx, uint32_t parity) -> bool {
        return __all_sync(0xffffffffu, mbar_wait(bar(idx), parity, abort_flag, limit));
      };
      const SmemDesc dq0 = sw128_desc_words(sbase + C::kOffQ, 16, 1024);
      const SmemDesc dk0 = sw128_desc_words(sbase + C::kOffK, 16, 1024);
      const SmemDesc dv0 = sw128_desc_words(sbase + C::kOffV, C::kBoxBytes, 1024);
      auto issue_qk = [&](int j) {   // S_{j&1} = Q K_j^T, K_j in stage j % kStages
        const int sb = j & 1, kst = j % C::kStages;
        const SmemDesc dk = desc_step(dk0, kst * C::kKTileBytes);
#pragma unroll
        for (int kk = 0; kk < DH / 16; ++kk) {
          const uint32_t off = (kk >> 2) * C::kBoxBytes + (kk & 3) * 32;
          umma_ss_we(tmem + 128 * sb, desc_step(dq0, off), desc_step(dk, off), kIdQK, kk > 0 ? 1u : 0u);
        }
        umma_commit_we(bar(C::kBarSFull + sb));
        umma_commit_we(bar(C::kBarKEmpty + kst));
      };
      // Scores run one key tile ahead: QK(j+1) is in its own buffer while
      // the softmax works on tile j, and QK(j+2) goes in right behind PV(j),
      // which has read P(j) out of the buffer QK(j+2) overwrites.
      bool ok = wait1(C::kBarQReady, 0);
      for (int j = 0; j < 2 && j < n && ok; ++j) {
        ok = wait1(C::kBarKFull + j % C::kStages, static_cast<uint32_t>((j / C::kStages) & 1));
        if (!ok) break;
        tc_fence_after_sync();
        issue_qk(j);
      }
      for (int j = 0; j < n && ok; ++j) {
        const int sb = j & 1, vst = j % C::kStages;
        ok = wait1(C::kBarPReady + sb, static_cast<uint32_t>((j >> 1) & 1)) &&
             wait1(C::kBarVReady + vst, static_cast<uint32_t>((j / C::kStages) & 1));
        if (!ok) break;
        tc_fence_after_sync();
        const SmemDesc dv = desc_step(dv0, vst * C::kVTileBytes);
#pragma unroll
        for (int kk = 0; kk < kTileN / 16; ++kk)
          umma_ts_we(tmem + C::kTO, tmem + 128 * sb + kk * 8, desc_step(dv, kk * 2048), kIdPV,
                     (j > 0 || kk > 0) ? 1u : 0u);
        umma_commit_we(bar(C::kBarVEmpty + vst));
        umma_commit_we(bar(C::kBarPVDone));
        if (j == n - 1) umma_commit_we(bar(C::kBarOFull));
        if (j + 2 < n) {
          ok = wait1(C::kBarKFull + (j + 2) % C::kStages, static_cast<uint32_t>(((j + 2) / C::kStages) & 1));
          if (!ok) break;
          tc_fence_after_sync();
          issue_qk(j + 2);
        }
      }
      int no_abort = 0;
      umma_commit_we(bar(C::kBarDrain));
      mbar_wait(bar(C::kBarDrain), 0, &no_abort, limit);
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ============================== softmax =============================
    const uint32_t quad = warp & 3;
    const int row = static_cast<int>(quad * 32 + lane);
    const bool valid = row < rows_valid;
    const int hh = valid ? row / n_q : 0;
    const int i = valid ? row - hh * n_q : 0;
    // Rows outside the tile's valid range see nothing.
    const int64_t lim = valid ? row_key_limit(p.mask, p.sh.n_k, b, i) : 0;
    const uint32_t lane_base = (quad * 32u) << 16;
    const uint32_t tO = tmem + lane_base + C::kTO;
    const float sl2 = p.scale_log2;
    float m_ref = -INFINITY;   // reference maximum, exp2 domain (lazy, as in the forward kernel)
    float l_sum = 0.f;         // sum of the weights (for the LSE)
    float l_used = 0.f;        // sum of the bf16-rounded weights the PV product used
    bool ok = *abort_flag == 0;
    uint32_t rr[32];
    for (int j = 0; j < n && ok; ++j) {
      const int st = j & 1;
      const uint32_t tS = tmem + lane_base + 128 * st;
      ok = __all_sync(0xffffffffu, mbar_wait(bar(C::kBarSFull + st), static_cast<uint32_t>((j >> 1) & 1), abort_flag,
                                             limit));
      if (!ok) break;
      tc_fence_after_sync();
      uint32_t sc[4][32];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld32_nowait(tS + c * 32, sc[c]);
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_wait_ld32(sc[c]);
      const int64_t lrel64 = lim - static_cast<int64_t>(t0 + j) * kTileN;
      const int lim_rel = lrel64 > kTileN ? kTileN : (lrel64 < 0 ? 0 : static_cast<int>(lrel64));
      if (__any_sync(0xffffffffu, lim_rel < kTileN)) {
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int k = 0; k < 32; ++k)
            sc[c][k] = (c * 32 + k < lim_rel) ? sc[c][k] : __float_as_uint(-INFINITY);
      }
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
        // (A row that has seen no visible key yet has m_ref = -inf and gets
        // alpha = 0, which rescales its all-zero sums and O.)
        const bool need = m_new > m_ref + 8.0f;
        if (__any_sync(0xffffffffu, need)) {
          // O must be settled: PV(j-1) done.
          ok = __all_sync(0xffffffffu, mbar_wait(bar(C::kBarPVDone), static_cast<uint32_t>((j - 1) & 1),
                                                 abort_flag, limit));
          if (!ok) break;
          tc_fence_after_sync();
          const float alpha = need ? fast_exp2(m_ref - m_new) : 1.0f;
          if (need) {
            l_sum *= alpha;
            l_used *= alpha;
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
      const float nm = (m_ref == -INFINITY) ? 0.f : -m_ref;
      float ls[2][2] = {{0.f, 0.f}, {0.f, 0.f}}, lu[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t pw[16];
#pragma unroll
        for (int k = 0; k < 32; k += 2) {
          float x0, x1;
          ffma2(x0, x1, __uint_as_float(sc[c][k]), __uint_as_float(sc[c][k + 1]), sl2, sl2, nm, nm);
          const float p0 = fast_exp2(x0), p1 = fast_exp2(x1);
          const uint32_t pk = pack_bf16x2(p0, p1);
          fadd2(ls[c & 1][0], ls[c & 1][1], p0, p1);
          fadd2(lu[c & 1][0], lu[c & 1][1], bf16_lo(pk), bf16_hi(pk));
          pw[k >> 1] = pk;
        }
        tmem_st16_nowait(tS + c * 16, pw);
      }
      l_sum += (ls[0][0] + ls[0][1]) + (ls[1][0] + ls[1][1]);
      l_used += (lu[0][0] + lu[0][1]) + (lu[1][0] + lu[1][1]);
      tmem_wait_st();
      tc_fence_before_sync();
      mbar_arrive(bar(C::kBarPReady + st));
    }

    // ---- epilogue ----
    if (ok && n > 0) {
      // The scores of tile n-1 imply only PV(n-3) done (QK(n-1) followed it),
      // so PV(n-2) and PV(n-1) may both be pending, and a parity wait on the
      // PV-done barrier could match the phase before them: the last product
      // has a barrier of its own.
      ok = __all_sync(0xffffffffu, mbar_wait(bar(C::kBarOFull), 0, abort_flag, limit));
      tc_fence_after_sync();
    }
    if (ok) {
      const int64_t qrow = valid ? (static_cast<int64_t>(b * p.sh.Hq + hkv * p.sh.group + h0 + hh) * n_q + i) : 0;
      const float inv_l = l_used > 0.f ? 1.0f / l_used : 0.f;
      // LSE of this key range (natural log); -inf when the range holds no
      // visible key of this row.
      const float lse = l_sum > 0.f ? (m_ref + fast_log2(l_sum)) * kLn2 : -INFINITY;
      if (p.nsplit == 1) {
        const int64_t row_off = qrow * DV;
        uint4* orow = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.O) + row_off);
        uint4* lorow = p.O_lo ? reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.O_lo) + row_off) : nullptr;
#pragma unroll
        for (int c = 0; c < DV / 32; ++c) {
          if (n > 0) tmem_ld32(tO + c * 32, rr);
          uint32_t wo[16], lo[16];
#pragma unroll
          for (int k = 0; k < 32; k += 2) {
            const float o0 = n > 0 ? __uint_as_float(rr[k]) * inv_l : 0.f;
            const float o1 = n > 0 ? __uint_as_float(rr[k + 1]) * inv_l : 0.f;
            wo[k >> 1] = pack_bf16x2(o0, o1);
            lo[k >> 1] = pack_bf16x2(o0 - bf16_lo(wo[k >> 1]), o1 - bf16_hi(wo[k >> 1]));
          }
          if (valid) {
#pragma unroll
            for (int v = 0; v < 4; ++v)
              orow[c * 4 + v] = make_uint4(wo[4 * v], wo[4 * v + 1], wo[4 * v + 2], wo[4 * v + 3]);
            if (lorow) {
#pragma unroll
              for (int v = 0; v < 4; ++v)
                lorow[c * 4 + v] = make_uint4(lo[4 * v], lo[4 * v + 1], lo[4 * v + 2], lo[4 * v + 3]);
            }
          }
        }
        if (valid) p.LSE[qrow] = lse;
      } else {
        // Partial output of this key range (normalised within the range)
        // and its log-sum-exp, for the merge kernel.
        const int64_t rows_total = static_cast<int64_t>(p.sh.B) * p.sh.Hq * n_q;
        float4* orow = reinterpret_cast<float4*>(p.Opart + (split * rows_total + qrow) * DV);
#pragma unroll
        for (int c = 0; c < DV / 32; ++c) {
          if (n > 0) tmem_ld32(tO + c * 32, rr);
          if (valid) {
#pragma unroll
            for (int v = 0; v < 8; ++v)
              orow[c * 8 + v] =
                  n > 0 ? make_float4(__uint_as_float(rr[4 * v]) * inv_l, __uint_as_float(rr[4 * v + 1]) * inv_l,
                                      __uint_as_float(rr[4 * v + 2]) * inv_l, __uint_as_float(rr[4 * v + 3]) * inv_l)
                        : make_float4(0.f, 0.f, 0.f, 0.f);
          }
        }
        if (valid) p.Lpart[split * rows_total + qrow] = lse;
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

// Merge of the key-range partials: one warp per query row.
//   LSE = M + ln sum_s exp(LSE_s - M),  O = sum_s exp(LSE_s - LSE) O_s,
// with M = max_s LSE_s (ranges without a visible key have LSE_s = -inf and
// weight 0).
template <int DV>
__global__ void __launch_bounds__(256)
attn_decode_merge_kernel(int64_t rows, int nsplit, const float* __restrict__ Opart, const float* __restrict__ Lpart,
                         __nv_bfloat16* __restrict__ O, __nv_bfloat16* __restrict__ O_lo, float* __restrict__ LSE) {
  const int64_t r = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  if (r >= rows) return;
  const uint32_t lane = threadIdx.x & 31;
  float M = -INFINITY;
  for (int s = 0; s < nsplit; ++s) M = fmaxf(M, Lpart[s * rows + r]);
  constexpr int kPer = DV / 32;   // elements per lane (2 or 4)
  float acc[kPer];
#pragma unroll
  for (int k = 0; k < kPer; ++k) acc[k] = 0.f;
  float wsum = 0.f;
  for (int s = 0; s < nsplit; ++s) {
    const float ls = Lpart[s * rows + r];
    const float w = (ls == -INFINITY) ? 0.f : fast_exp2((ls - M) * kLog2e);
    wsum += w;
    const float* src = Opart + (s * rows + r) * DV + lane * kPer;
#pragma unroll
    for (int k = 0; k < kPer; ++k) acc[k] = fmaf(w, src[k], acc[k]);
  }
  const float inv = wsum > 0.f ? 1.0f / wsum : 0.f;
  __nv_bfloat16* orow = O + r * DV + lane * kPer;
#pragma unroll
  for (int k = 0; k < kPer; k += 2) {
    const float o0 = acc[k] * inv, o1 = acc[k + 1] * inv;
    const uint32_t w = pack_bf16x2(o0, o1);
    *reinterpret_cast<uint32_t*>(orow + k) = w;
    if (O_lo) *reinterpret_cast<uint32_t*>(O_lo + r * DV + lane * kPer + k) =
        pack_bf16x2(o0 - bf16_lo(w), o1 - bf16_hi(w));
  }
  if (lane == 0) LSE[r] = M + fast_log2(wsum) * kLn2;
}

template <int DH, int DV>
cudaError_t launch_decode_t(const CUtensorMap& tmK, const CUtensorMap& tmV, const DecParams& p, cudaStream_t stream) {
  using C = DecCfg<DH, DV>;
  auto kern = attn_decode_kernel<DH, DV>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (e != cudaSuccess) return e;
  dim3 grid(static_cast<unsigned>(p.sh.B * p.sh.Hkv * p.chunks), static_cast<unsigned>(p.nsplit));
  kern<<<grid, C::kThreads, C::kSmemBytes, stream>>>(tmK, tmV, p);
  e = cudaGetLastError();
  if (e != cudaSuccess || p.nsplit == 1) return e;
  const int64_t rows = static_cast<int64_t>(p.sh.B) * p.sh.Hq * p.sh.n_q;
  attn_decode_merge_kernel<DV><<<static_cast<unsigned>((rows + 7) / 8), 256, 0, stream>>>(
      rows, p.nsplit, p.Opart, p.Lpart, static_cast<__nv_bfloat16*>(p.O), static_cast<__nv_bfloat16*>(p.O_lo),
      p.LSE);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attn_decode(int dh, int dv, const CUtensorMap& tmK, const CUtensorMap& tmV, const DecParams& p,
                               cudaStream_t stream) {
  if (dh == 128 && dv == 128) return launch_decode_t<128, 128>(tmK, tmV, p, stream);
  if (dh == 64 && dv == 64) return launch_decode_t<64, 64>(tmK, tmV, p, stream);
  if (dh == 128 && dv == 64) return launch_decode_t<128, 64>(tmK, tmV, p, stream);
  return cudaErrorInvalidValue;
}

}  // namespace esd
