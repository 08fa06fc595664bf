// attn_bwd_persist.cu -- the backward main kernel's persistent schedule on
// sm_103a: the same products, passes and precision as the grid kernel in
// attn_bwd.cu (which holds the formulas: "Appendix A.10 -- Attention
// matrices and backpropagation", eqs. A.10.5-A.10.9), with one CTA per SM
// taking (batch, KV head, 128-key tile) work items from a counter instead of
// one CTA per item.
//
// Why two schedules.  A CTA of the grid kernel spends about 18k cycles
// outside its steps (launch, barrier set-up, the K and V loads and their
// fp16 re-encoding, the pipeline's fill, the last dQ/dK products, the dK/dV
// epilogue), against about 5k cycles per 128-query step: a quarter of the
// time of an item with a few steps.  The persistent kernel hides most of it
// behind the neighbouring items' steps, but its steps run some 10-15 %
// slower (the roles' loops nest inside item loops, and the warps stall more
// often on instruction fetch), so the host takes it only for items of few
// steps (short query ranges, small head groups, causal MHA), and the grid
// kernel for long ones.
//
// Warp roles (512 threads), as in the grid kernel except where noted:
//   warp 0      TMA producer; also publishes the item numbers and claims
//               the next item about two steps before the current one ends.
//   warps 1, 3  MMA issuers.
//   warps 4-11  score warpgroups; at the start of every item all eight warps
//               re-encode its K and V tiles as fp16 (in the grid kernel the
//               read-out warps do), so that the read-out warps can finish
//               the previous item meanwhile.
//   warps 12-15 dQ read-out and the dK/dV epilogue.
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "bwd_scale.cuh"
#include "common.cuh"
#include "f16range.cuh"
#include "ptx.cuh"
#include "rotary.cuh"

namespace esd {
namespace {

template <int DH, int DV>
struct BwdPCfg {
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
  // The score warps' reduction over a work item: per warp w (8 warps)
  // red[4w .. 4w+3] = (largest |K| of its share of the tile, max ||v_j||,
  // max ||dO_i||, max |D_i|).
  static constexpr int kOffRed = kOffDd + kTileM * 4;
  // Work items: the two published item numbers, the score warps' copies of
  // them, and the read-out multipliers of two items in flight.
  static constexpr int kOffItem = kOffRed + 32 * 4;
  static constexpr int kOffItemScale = kOffItem + 16;
  // Per read-out warp: the fields of its current item it reads inside the
  // dQ loop (kept here rather than in registers, which the loop's 64
  // loaded columns need).
  static constexpr int kOffRo = kOffItemScale + 2 * 16;
  // The score warps' current item: its fields the step loop reads (kept
  // here rather than in registers, which the step's scores and weights
  // need).
  static constexpr int kOffScs = kOffRo + 4 * 64;
  static constexpr int kOffBar = kOffScs + 32;
  static constexpr int kBarKV = 0;
  static constexpr int kBarQFull = 1;                 // [2]
  static constexpr int kBarQEmpty = kBarQFull + 2;    // [2]
  static constexpr int kBarDOFull = kBarQEmpty + 2;
  static constexpr int kBarDOEmpty = kBarDOFull + 1;
  static constexpr int kBarK16 = kBarDOEmpty + 1;     // K tile re-encoded as fp16, multipliers published
  static constexpr int kBarV16 = kBarK16 + 1;         // V tile re-encoded as fp16
  static constexpr int kBarSFull = kBarV16 + 1;
  static constexpr int kBarDPFull = kBarSFull + 1;
  static constexpr int kBarPReady = kBarDPFull + 1;
  static constexpr int kBarDSReady = kBarPReady + 1;
  static constexpr int kBarDQFull = kBarDSReady + 1;
  static constexpr int kBarDQFree = kBarDQFull + 1;
  static constexpr int kBarDKDone = kBarDQFree + 1;   // dK(s) done: dS tile free again
  static constexpr int kBarDKDV = kBarDKDone + 1;     // the item's last dK, dV products done
  static constexpr int kBarKVFree = kBarDKDV + 1;     // the item's last dQ product done: K, V tiles free
  static constexpr int kBarAccFree = kBarKVFree + 1;  // the item's dK, dV read out of tensor memory
  static constexpr int kBarItemFull = kBarAccFree + 1;     // [2]
  static constexpr int kBarItemEmpty = kBarItemFull + 2;   // [2]
  static constexpr int kBarDrain = kBarItemEmpty + 2;
  static constexpr int kNumBars = kBarDrain + 1;
  // Readers of a published item number: the two MMA issuers, the score
  // warps' leader and the four read-out warps.
  static constexpr int kItemReaders = 7;
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

// The item's multipliers (bwd_scale.cuh), in one out-of-line copy.
__device__ __noinline__ CtaScale item_scale(float mv, float mdo, float md, float2 qo) {
  return cta_scale_of(mv, mdo, md, qo);
}

// A work item of the main kernel: the 128-key tile kt of (batch, KV head)
// bkv, with the z-th share of the group's query heads under a split.  Items
// are numbered with bkv fastest, then z, then kt, so that under a causal
// mask -- where the low key tiles see the most query tiles -- the costliest
// items come first and the CTAs that take items in number order finish
// close together.  Its steps run over the query heads of the share (outer)
// and the query tiles that can see its keys (inner).
struct BwdItem {
  int b, hkv, bkv, total, per_head, qt_first, head0;
  int64_t j0, klen, nq_b;
};

template <bool SPLIT>
__device__ __forceinline__ BwdItem bwd_item(int w, const BwdParams& p) {
  BwdItem it;
  const int bhkv = p.sh.B * p.sh.Hkv;
  const int zs = SPLIT ? p.hsplit : 1;
  const int kt = w / (bhkv * zs);
  const int r = w - kt * bhkv * zs;
  const int z = r / bhkv;
  it.bkv = r - z * bhkv;
  it.b = it.bkv / p.sh.Hkv;
  it.hkv = it.bkv - it.b * p.sh.Hkv;
  it.j0 = static_cast<int64_t>(kt) * kTileN;
  it.klen = key_len(p.mask, p.sh.n_k, it.b);
  it.nq_b = query_len(p.mask, p.sh.n_q, it.b);
  const int64_t i_first = first_row_seeing_key(p.mask, p.sh.n_q, p.sh.n_k, it.b, it.j0);
  const int nqt = static_cast<int>((it.nq_b + kTileM - 1) / kTileM);
  it.qt_first = i_first < it.nq_b ? static_cast<int>(i_first / kTileM) : 0;
  it.per_head = i_first < it.nq_b ? nqt - it.qt_first : 0;
  const int hps = SPLIT ? p.sh.group / p.hsplit : p.sh.group;
  it.total = it.per_head * hps;
  it.head0 = it.hkv * p.sh.group + (SPLIT ? z * hps : 0);
  return it;
}
// The same value through an opaque move: a role that decodes an item before
// and after a long loop re-decodes it from this copy instead of keeping
// every field in registers through the loop.
__device__ __forceinline__ int opaque_int(int x) {
  int y;
  asm volatile("mov.b32 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}
__device__ __forceinline__ int item_head(const BwdItem& it, int s) { return it.head0 + s / it.per_head; }
__device__ __forceinline__ int item_q0(const BwdItem& it, int s) { return (it.qt_first + s % it.per_head) * kTileM; }

// Persistent: a CTA per SM (or fewer when there are fewer items) takes work
// items from a counter until none are left (the first item of CTA c is c,
// each further one comes from an atomic add on the counter, which the
// backward's first stage zeroes).  The producer publishes each item number
// through a two-slot ring; every role walks the same items in the same
// order, and the barriers' phases run on over the whole sequence: per-step
// barriers on the global step count g, per-item barriers on the count of
// items with at least one step.  What overlaps at an item boundary: the
// next item's K and V tiles load as soon as the last dQ product has read
// the old ones, and the score warps re-encode them while the read-out warps
// read out the last dQ tile and write the finished item's dK and dV (whose
// tensor memory the next item's first dK and dV products wait for).
template <int DH, int DV, bool PACKED, bool ROPE, bool SPLIT>
__global__ void __launch_bounds__(512, 1)
attn_bwd_main_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                     const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                     const __grid_constant__ CUtensorMap tmdQ, const __grid_constant__ BwdParams p) {
  using C = BwdPCfg<DH, DV>;
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
  volatile int* item_s = reinterpret_cast<volatile int*>(smem + C::kOffItem);       // [2] published
  volatile int* dec_s = reinterpret_cast<volatile int*>(smem + C::kOffItem + 8);    // [2] score warps' copy
  float4* iscale_s = reinterpret_cast<float4*>(smem + C::kOffItemScale);            // [2] read-out multipliers

  const uint32_t warp = warp_id();
  const uint32_t lane = lane_id();

  if (threadIdx.x == 0) {
    mbar_init(bar(C::kBarKV), 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(C::kBarQFull + s), 1);
      mbar_init(bar(C::kBarQEmpty + s), 1);
      mbar_init(bar(C::kBarItemFull + s), 1);
      mbar_init(bar(C::kBarItemEmpty + s), C::kItemReaders);
    }
    mbar_init(bar(C::kBarDOFull), 1);
    mbar_init(bar(C::kBarDOEmpty), 1);
    mbar_init(bar(C::kBarK16), 256);
    mbar_init(bar(C::kBarV16), 256);
    mbar_init(bar(C::kBarSFull), 1);
    mbar_init(bar(C::kBarDPFull), 1);
    mbar_init(bar(C::kBarPReady), 256);
    mbar_init(bar(C::kBarDSReady), 256);
    mbar_init(bar(C::kBarDQFull), 1);
    mbar_init(bar(C::kBarDQFree), 128);
    mbar_init(bar(C::kBarDKDone), 1);
    mbar_init(bar(C::kBarDKDV), 2);    // one commit from each MMA issuer
    mbar_init(bar(C::kBarKVFree), 1);
    mbar_init(bar(C::kBarAccFree), 128);
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
  // Item k of this CTA, read by a whole warp from the ring (false: no item,
  // the producer stopped or a wait gave up); lane 0 releases the slot.
  auto read_item = [&](int k, int& w) -> bool {
    if (!wait_all(C::kBarItemFull + (k & 1), static_cast<uint32_t>((k >> 1) & 1))) return false;
    w = item_s[k & 1];
    __syncwarp();
    if (lane == 0) mbar_arrive(bar(C::kBarItemEmpty + (k & 1)));
    return w >= 0;
  };

  if (warp < 4) setmaxnreg_to<C::kRegsLow, C::kRegsLaunch>();
  if (warp == 0) {
    // =========================== TMA producer ===========================
    // Per item: the fp16 Q tile of its first step (into the two-stage
    // ring), the K and V tiles once the previous item's last dQ product has
    // read the old ones, the first dO tile; then per step a Q and a dO tile.
    if (lane == 0) {
      bool ok = *abort_flag == 0;
      if (ok) {
        tma_prefetch_map(&tmQ);
        tma_prefetch_map(&tmK);
        tma_prefetch_map(&tmV);
        tma_prefetch_map(&tmdO);
      }
      int q_issued[2] = {0, 0}, do_issued = 0, kv_issued = 0;
      int g = 0, ka = 0;
      int cur = ok ? static_cast<int>(blockIdx.x) : -1;
      // Warm L2 with the Q and dO tiles of query tile qt of head hd.
      auto prefetch_at = [&](int b, int hd, int qt) {
        const TmaYZ yz = q_tma(PACKED, p.lay, p.sh.Hq, b, hd, qt * kTileM);
        for (int c = 0; c < DH / 64; ++c) tma_prefetch_l2_3d(&tmQ, c * 64, yz.y, yz.z);
        for (int c = 0; c < DV / 64; ++c) tma_prefetch_l2_3d(&tmdO, c * 64, yz.y, yz.z);
      };
      for (int k = 0;; ++k) {
        if (k >= 2 && !mbar_wait(bar(C::kBarItemEmpty + (k & 1)), static_cast<uint32_t>(((k >> 1) - 1) & 1),
                                 abort_flag, limit)) {
          ok = false;
          break;
        }
        item_s[k & 1] = cur;
        mbar_arrive(bar(C::kBarItemFull + (k & 1)));
        if (cur < 0) break;
        const BwdItem it = bwd_item<SPLIT>(cur, p);
        // The next item is claimed late -- once this item's last tiles are
        // requested, about two steps before it ends -- so that items go to
        // whichever CTA frees first, in number order (costliest first).
        int nxt = -1;
        bool claimed = false;
        auto claim = [&]() {
          nxt = static_cast<int>(atomicAdd(p.work_ctr, 1u)) + static_cast<int>(gridDim.x);
          if (nxt >= p.nitems) nxt = -1;
          claimed = true;
          if (nxt < 0) return;
          // Its K and V tiles and first two Q, dO tiles into L2 while this
          // item ends.
          const BwdItem nx = bwd_item<SPLIT>(nxt, p);
          if (nx.total == 0) return;
          const TmaYZ nyz = k_tma(PACKED, p.lay, p.sh.Hkv, nx.b, nx.hkv, static_cast<int>(nx.j0));
          for (int c = 0; c < DH / 64; ++c) tma_prefetch_l2_3d(&tmK, c * 64, nyz.y, nyz.z);
          for (int c = 0; c < DV / 64; ++c) tma_prefetch_l2_3d(&tmV, c * 64, nyz.y, nyz.z);
          prefetch_at(nx.b, nx.head0, nx.qt_first);
          if (nx.total > 1)
            prefetch_at(nx.b, nx.per_head > 1 ? nx.head0 : nx.head0 + 1, nx.per_head > 1 ? nx.qt_first + 1 : nx.qt_first);
        };
        if (it.total > 0) {
          // Step s is query tile qt of head hd: the item's tiles
          // [qt_first, qt_end) of each of its heads in turn.
          const int qt_end = it.qt_first + it.per_head;
          int qt = it.qt_first, hd = it.head0;
          int qt2 = qt, hd2 = hd;   // step s + 2
          for (int a = 0; a < 2; ++a) {
            if (++qt2 == qt_end) {
              qt2 = it.qt_first;
              ++hd2;
            }
          }
          for (int s = 0; s < it.total; ++s, ++g) {
            const int st = g & 1;
            const TmaYZ yz = q_tma(PACKED, p.lay, p.sh.Hq, it.b, hd, qt * kTileM);
            if (!mbar_wait(bar(C::kBarQEmpty + st), static_cast<uint32_t>(((g >> 1) & 1) ^ 1), abort_flag, limit)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(bar(C::kBarQFull + st), C::kQTileBytes);
            for (int c = 0; c < DH / 64; ++c)
              tma_load_3d(sbase + C::kOffQ + st * C::kQTileBytes + c * C::kBlockBytes, &tmQ,
                          bar(C::kBarQFull + st), c * 64, yz.y, yz.z);
            ++q_issued[st];
            if (s == 0) {
              if (ka > 0 && !mbar_wait(bar(C::kBarKVFree), static_cast<uint32_t>((ka - 1) & 1), abort_flag, limit)) {
                ok = false;
                break;
              }
              const TmaYZ kyz = k_tma(PACKED, p.lay, p.sh.Hkv, it.b, it.hkv, static_cast<int>(it.j0));
              mbar_arrive_expect_tx(bar(C::kBarKV), C::kKTileBytes + C::kVTileBytes);
              for (int c = 0; c < DH / 64; ++c)
                tma_load_3d(sbase + C::kOffK + c * C::kBlockBytes, &tmK, bar(C::kBarKV), c * 64, kyz.y, kyz.z);
              for (int c = 0; c < DV / 64; ++c)
                tma_load_3d(sbase + C::kOffV + c * C::kBlockBytes, &tmV, bar(C::kBarKV), c * 64, kyz.y, kyz.z);
              ++kv_issued;
            }
            // One dO stage: dO(g) is read by dP(g) and dV(g) only, so the
            // next tile loads as soon as dV(g) is done, well before dP(g+1).
            if (g > 0 && !mbar_wait(bar(C::kBarDOEmpty), static_cast<uint32_t>((g - 1) & 1), abort_flag, limit)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(bar(C::kBarDOFull), C::kDOTileBytes);
            for (int c = 0; c < DV / 64; ++c)
              tma_load_3d(sbase + C::kOffDO + c * C::kBlockBytes, &tmdO, bar(C::kBarDOFull), c * 64, yz.y, yz.z);
            ++do_issued;
            if (s + 1 == it.total) claim();
            // Warm L2 with the tiles two steps ahead: their shared-memory
            // stage is only free once the step before has finished, which
            // leaves too little time to hide a load from HBM.
            if (s + 2 < it.total) prefetch_at(it.b, hd2, qt2);
            if (++qt == qt_end) {
              qt = it.qt_first;
              ++hd;
            }
            if (++qt2 == qt_end) {
              qt2 = it.qt_first;
              ++hd2;
            }
          }
          if (!ok) break;
          ++ka;
        }
        if (!claimed) claim();
        cur = nxt;
      }
      if (*abort_flag) {
        // Let every load already issued land before the CTA can exit.
        int no_abort = 0;
        if (kv_issued) mbar_wait(bar(C::kBarKV), static_cast<uint32_t>((kv_issued - 1) & 1), &no_abort, limit);
        for (int st = 0; st < 2; ++st) {
          if (q_issued[st])
            mbar_wait(bar(C::kBarQFull + st), static_cast<uint32_t>((q_issued[st] - 1) & 1), &no_abort, limit);
        }
        if (do_issued) mbar_wait(bar(C::kBarDOFull), static_cast<uint32_t>((do_issued - 1) & 1), &no_abort, limit);
      }
    }
  } else if (warp == 1 || warp == 3) {
    // =========================== MMA issuers ============================
    // Two issuers on two SM sub-partitions split each step's products:
    //   warp 1 (A):  dV(g) | S(g+1) -> X | dP(g+1) -> Y
    //   warp 3 (B):  dQ(g) -> Y, dK(g)
    // An MMA issue takes several instructions of the issuing thread, and the
    // score and read-out warps sharing a sub-partition leave it only part of
    // the issue slots; two issuers halve the instructions each one needs.
    // Ordering across the two (g counts steps over all of the CTA's items):
    //   X: dV(g) reads P^T(g) before S(g+1) overwrites it (both A, in order).
    //   Y: dP(g) [A] -> score warps read it -> dQ(g) [B, after dS ready]
    //      -> read-out -> dP(g+1) [A, after dQ free].
    //   dS tile: dQ(g), dK(g) [B] read it; the score warps rewrite it only
    //      after dP(g+1) has landed, and A issues dP(g+1) after B's dK(g)
    //      has completed.
    //   Q(g) stage: S(g) [A] completed before the scores of step g were
    //      seen, so B's commit after dK(g) releases it.
    //   K, V tiles: B's commit after an item's last dQ releases them (S and
    //      dP of that step completed before its dS was written).
    //   dK, dV accumulators: an item's first dV [A] and dK [B] wait until
    //      the read-out warps have taken the previous item's sums out.
    // Each issuer warp runs converged: all lanes wait (with a vote) and one
    // elected lane issues, so that descriptors and tensor-memory addresses
    // stay warp-uniform and the issue keeps its rate under the score warps'
    // pressure.
    const bool issuer_a = warp == 1;
    bool ok = __all_sync(0xffffffffu, *abort_flag == 0);
    constexpr uint32_t kIdS = idesc_f16_f32(128, 128, false, false);    // S^T = K Q^T (fp16)
    constexpr uint32_t kIdDP = idesc_f16_f32(128, 128, false, false);   // dP^T = V dO^T (fp16)
    constexpr uint32_t kIdDV = idesc_f16_f32(128, DV, false, true);     // dV += P^T dO (fp16)
    constexpr uint32_t kIdDK = idesc_f16_f32(128, DH, false, true);     // dK += dS^T Q
    constexpr uint32_t kIdDQ = idesc_f16_f32(128, DH, true, true);      // dQ = dS K
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
    auto issue_s = [&](int g) {   // S^T = K Q^T -> X
      const SmemDesc dq = desc_step(dQ_k, (g & 1) * C::kQTileBytes);
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
    int g = 0, ka = 0;
    for (int k = 0; ok; ++k) {
      int w = -1;
      if (!read_item(k, w)) break;
      const BwdItem it = bwd_item<SPLIT>(w, p);
      if (it.total == 0) continue;
      const uint32_t pk = static_cast<uint32_t>(ka & 1);
      if (issuer_a) {
        ok = wait_all(C::kBarK16, pk);
        if (ok) ok = wait_all(C::kBarQFull + (g & 1), static_cast<uint32_t>((g >> 1) & 1));
        if (ok) {
          tc_fence_after_sync();
          issue_s(g);
        }
        if (ok) ok = wait_all(C::kBarDOFull, static_cast<uint32_t>(g & 1));
        if (ok) ok = wait_all(C::kBarV16, pk);
        if (ok && g > 0) ok = wait_all(C::kBarDQFree, static_cast<uint32_t>((g - 1) & 1));
        if (ok && g > 0) ok = wait_all(C::kBarDKDone, static_cast<uint32_t>((g - 1) & 1));
        if (ok) {
          tc_fence_after_sync();
          issue_dp();
        }
        for (int s = 0; s < it.total && ok; ++s) {
          const int gs = g + s;
          ok = wait_all(C::kBarPReady, static_cast<uint32_t>(gs & 1));
          if (ok && s == 0 && ka > 0) ok = wait_all(C::kBarAccFree, static_cast<uint32_t>((ka - 1) & 1));
          if (!ok) break;
          tc_fence_after_sync();
#pragma unroll 1
          for (int kk = 0; kk < kTileM / 16; ++kk)
            umma_ts_we(tmem + C::kTdV, tmem + C::kTX + half_col(kk), desc_step(dDO_mn, kk * 2048), kIdDV,
                      (s > 0 || kk > 0) ? 1u : 0u);
          umma_commit_we(bar(C::kBarDOEmpty));   // dP(g) and dV(g) were dO(g)'s only readers
          if (s + 1 < it.total) {
            ok = wait_all(C::kBarQFull + ((gs + 1) & 1), static_cast<uint32_t>(((gs + 1) >> 1) & 1));
            if (!ok) break;
            tc_fence_after_sync();
            issue_s(gs + 1);
            ok = wait_all(C::kBarDOFull, static_cast<uint32_t>((gs + 1) & 1));
            if (ok) ok = wait_all(C::kBarDQFree, static_cast<uint32_t>(gs & 1));
            if (ok) ok = wait_all(C::kBarDKDone, static_cast<uint32_t>(gs & 1));
            if (!ok) break;
            tc_fence_after_sync();
            issue_dp();
          }
        }
      } else {
        for (int s = 0; s < it.total && ok; ++s) {
          const int gs = g + s;
          ok = wait_all(C::kBarDSReady, static_cast<uint32_t>(gs & 1));
          if (!ok) break;
          tc_fence_after_sync();
          // dQ(g) first, into Y (the score warps have read dP^T out of it),
          // so that its read-out overlaps dK(g); both take dS from the
          // shared-memory buffer, as the MN-major (dQ) and the K-major (dK)
          // view of the same swizzled tile.
#pragma unroll 1
          for (int kk = 0; kk < kTileN / 16; ++kk)
            umma_ss_we(tmem + C::kTY, desc_step(dDS_mn, kk * 2048), desc_step(dK_mn, kk * 2048), kIdDQ,
                      kk > 0 ? 1u : 0u);
          umma_commit_we(bar(C::kBarDQFull));
          if (s + 1 == it.total) umma_commit_we(bar(C::kBarKVFree));
          if (s == 0 && ka > 0) {
            ok = wait_all(C::kBarAccFree, static_cast<uint32_t>((ka - 1) & 1));
            if (!ok) break;
            tc_fence_after_sync();
          }
#pragma unroll 1
          for (int kk = 0; kk < kTileM / 16; ++kk)
            umma_ss_we(tmem + C::kTdK, desc_step(dDS_k, (kk >> 2) * C::kBlockBytes + (kk & 3) * 32),
                      desc_step(dQ_mn, (gs & 1) * C::kQTileBytes + kk * 2048), kIdDK, (s > 0 || kk > 0) ? 1u : 0u);
          umma_commit_we(bar(C::kBarQEmpty + (gs & 1)));
          umma_commit_we(bar(C::kBarDKDone));
        }
      }
      if (!ok) break;
      umma_commit_we(bar(C::kBarDKDV));
      g += it.total;
      ++ka;
    }
    int no_abort = 0;
    umma_commit_we(bar(C::kBarDrain));
    mbar_wait(bar(C::kBarDrain), 0, &no_abort, limit);
    __syncwarp();
  } else if (warp >= 4 && warp < 12) {
    // =========================== score warpgroups =======================
    // Two warpgroups: h = 0 takes query columns [0, 64), h = 1 [64, 128);
    // in both, thread = key row = TMEM lane.  At the start of an item all
    // eight warps re-encode its K and V tiles as fp16.
    setmaxnreg_to<C::kRegsScore, C::kRegsLaunch>();
    const int h = static_cast<int>(warp - 4) / 4;
    const uint32_t quad = warp & 3;
    const int jj = static_cast<int>(quad * 32 + lane);
    const int tid = static_cast<int>(threadIdx.x) - 128 - 128 * h;
    const int ts = static_cast<int>(threadIdx.x) - 128;   // 0 .. 255 over both warpgroups
    const uint32_t lane_base = (quad * 32u) << 16;
    const uint32_t tX = tmem + lane_base + C::kTX;
    const uint32_t tY = tmem + lane_base + C::kTY;
    uint8_t* ds_row = smem + C::kOffDS + h * C::kBlockBytes + jj * 128;
    const uint32_t wg_bar = 1 + static_cast<uint32_t>(h);
    constexpr uint32_t kAllBar = 4;   // the 256 score threads
    volatile int* scs = reinterpret_cast<volatile int*>(smem + C::kOffScs);
    bool ok = *abort_flag == 0;
    // The weights P of this thread's 64 columns, kept in fp32 from the P pass
    // for the dS pass (the fp16 copy goes to tensor memory for dV).
    float pf[64];
    int g = 0, ka = 0;
    // Every score thread passes the same named barriers in the same order:
    // one per item (the leader's copy of the item number is read after it),
    // one more per item with steps (the reduction), and two per step, even
    // after a wait has given up (the work is then skipped), so that no warp
    // can be left waiting at one.
    for (int k = 0;; ++k) {
      if (ts == 0) {
        int w = -1;
        if (*abort_flag == 0 &&
            mbar_wait(bar(C::kBarItemFull + (k & 1)), static_cast<uint32_t>((k >> 1) & 1), abort_flag, limit)) {
          w = item_s[k & 1];
          mbar_arrive(bar(C::kBarItemEmpty + (k & 1)));
        }
        dec_s[k & 1] = w;
      }
      __syncwarp();
      named_bar_sync(kAllBar, 256);
      const int w = dec_s[k & 1];
      if (w < 0) break;
      const BwdItem it = bwd_item<SPLIT>(w, p);
      if (it.total == 0) continue;
      const uint32_t pk = static_cast<uint32_t>(ka & 1);
      auto step_head = [&](int s) { return item_head(it, s); };
      auto step_q0 = [&](int s) { return item_q0(it, s); };
      const int jrow = static_cast<int>(it.j0) + jj;
      const bool row_masked = jrow >= it.klen;
      // The step loop's item fields, published by the reduction barrier
      // below (every reader of the previous item's passed this item's
      // first barrier).
      if (ts == 0) {
        scs[0] = it.b;
        scs[1] = static_cast<int>(it.nq_b);
        scs[2] = it.qt_first;
        scs[3] = it.per_head;
        scs[4] = it.head0;
        scs[5] = it.total;
        scs[6] = p.mask.causal ? static_cast<int>(causal_offset(p.mask, it.b)) : 0;
        scs[7] = g;
      }
      // This thread's -LSE log2(e) and -D entries (query q0 + 64h + tid, for
      // tid < 64) of a step, loaded one step ahead so the global latency is
      // off the critical path.  Both are kept negated so that one paired
      // fused multiply-add forms x sl2 - LSE log2(e) and dP_acc cp - D dmul.
      // (b, nq, head, q0): the step's batch element, its sequence's query
      // count, head and first query row.
      auto row_terms = [&](int b, int nq, int head, int q0, float& nlse2, float& nd) {
        const int i = q0 + 64 * h + tid;
        // Query rows past the sequence get LSE = -inf: their weights P, and so
        // their dS and contributions to dK, dV, dQ, are exactly 0.
        const bool in = tid < 64 && i < nq;
        const int64_t r = in ? q_vec(PACKED, p.lay, p.sh.Hq, p.sh.n_q, b, head, i) : 0;
        nlse2 = in ? -p.LSE[r] * kLog2e : -INFINITY;
        nd = in ? -p.D[r] : 0.f;
      };
      auto load_row_terms = [&](int s, float& nlse2, float& nd) {   // (prologue: from the item itself)
        row_terms(it.b, static_cast<int>(it.nq_b), step_head(s), step_q0(s), nlse2, nd);
      };
      auto slot_row_terms = [&](int s, float& nlse2, float& nd) {   // (step loop: from the slot)
        const int ph = scs[3];
        row_terms(scs[0], scs[1], scs[4] + s / ph, (scs[2] + s % ph) * kTileM, nlse2, nd);
      };
      float lse_next = 0.f, d_next = 0.f;
      if (ok) load_row_terms(0, lse_next, d_next);
      // ---- the item's K and V tiles as fp16, and its multipliers ----
      // Largest |K| over the tile (rows inside kv_len), the V rows' norms
      // and every step's tile maxima, reduced over the eight warps; then K
      // and V re-encoded in place: rows in [kv_len, n_k) hold caller memory
      // that may be anything (even NaN) and become zeros -- their dS
      // entries are 0, but 0 * NaN would still poison dQ.  Rows at or
      // beyond n_k arrive as zeros from the TMA bounds check.
      constexpr int kKc = C::kKTileBytes / 16 / 256;
      constexpr int kVc = C::kVTileBytes / 16 / 256;
      auto tile_row = [](int k) { return (k % (C::kBlockBytes / 16)) / 8; };   // 8 chunks per 128-byte row
      uint4* kt = reinterpret_cast<uint4*>(smem + C::kOffK);
      uint4* vt = reinterpret_cast<uint4*>(smem + C::kOffV);
      if (ok) ok = wait_all(C::kBarKV, pk);
      uint32_t km = 0u;
      float vn2 = 0.f, mdo = 0.f, md = 0.f;
      // (The per-item loops stay mostly rolled: the kernel's code has to fit
      // the instruction cache next to the step loops.)
      if (ok) {
#pragma unroll 2
        for (int i = 0; i < kKc; ++i) {
          const uint4 u = kt[ts + 256 * i];
          if (it.j0 + tile_row(ts + 256 * i) < it.klen) km = bf16_absmax_fold(km, u);
        }
        if (h == 0 && !row_masked) {
#pragma unroll 1
          for (int c = 0; c < DV / 64; ++c) {
#pragma unroll 2
            for (int q = 0; q < 8; ++q) {
              const uint4 u = *reinterpret_cast<const uint4*>(smem + C::kOffV + c * C::kBlockBytes + jj * 128 + q * 16);
              const uint32_t wv[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                vn2 = fmaf(bf16_lo(wv[e]), bf16_lo(wv[e]), vn2);
                vn2 = fmaf(bf16_hi(wv[e]), bf16_hi(wv[e]), vn2);
              }
            }
          }
        }
#pragma unroll 1
        for (int idx = ts; idx < it.total; idx += 256) {
          const int bhq = it.b * p.sh.Hq + step_head(idx);
          const float4 t = p.tilemax[static_cast<int64_t>(bhq) * p.nqt + step_q0(idx) / kTileM];
          mdo = fmaxf(mdo, t.x);
          md = fmaxf(md, t.y);
        }
      }
      float kmax = bf16_absmax_value(km), mv = sqrtf(vn2);
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        kmax = fmaxf(kmax, __shfl_xor_sync(0xffffffffu, kmax, off));
        mv = fmaxf(mv, __shfl_xor_sync(0xffffffffu, mv, off));
        mdo = fmaxf(mdo, __shfl_xor_sync(0xffffffffu, mdo, off));
        md = fmaxf(md, __shfl_xor_sync(0xffffffffu, md, off));
      }
      const int wi = static_cast<int>(warp) - 4;
      if (lane == 0) {
        red_s[4 * wi] = kmax;
        red_s[4 * wi + 1] = mv;
        red_s[4 * wi + 2] = mdo;
        red_s[4 * wi + 3] = md;
      }
      __syncwarp();
      named_bar_sync(kAllBar, 256);   // also: every read of the bf16 tiles is done
#pragma unroll
      for (int x = 0; x < 8; ++x) {
        kmax = fmaxf(kmax, red_s[4 * x]);
        mv = fmaxf(mv, red_s[4 * x + 1]);
        mdo = fmaxf(mdo, red_s[4 * x + 2]);
        md = fmaxf(md, red_s[4 * x + 3]);
      }
      // The item's multipliers (CtaScale): the scores come out of S^T =
      // K16 Q16^T as 2^(k + q) S_raw, so P = exp2(S_acc sl2 - LSE log2e)
      // with sl2 = scale log2e 2^-(k + q); and dS' = 2^g dS =
      // P (dP_acc cp + (-D) dmul) with cp = 2^(g - o - v), dmul = 2^g.
      float sl2 = p.scale_log2, cp = 1.f, dmul = 1.f;
      if (ok) {
        int kexp = f16_tile_exponent(kmax);
        if (kexp == kExpZero) kexp = 0;
        const CtaScale cs = item_scale(mv, mdo, md, p.grpexp[it.bkv]);
        if (ts == 0) {
          if (f16_saturates(kmax, kexp) || f16_saturates(cs.mv, cs.v) || cs.overflow)
            record_status(p.status, ATTN_ERR_RANGE);
          // For the read-out warps: dQ_acc = 2^(g + k) dS K, dK_acc =
          // 2^(g + q) dS^T Q, dV_acc = 2^o dV.
          iscale_s[pk] = make_float4(exp2_int(-cs.g - kexp), p.scale * exp2_int(-cs.g - cs.q), exp2_int(-cs.o), 0.f);
        }
        const float ks = exp2_int(kexp);
#pragma unroll 2
        for (int i = 0; i < kKc; ++i) {
          const int e = ts + 256 * i;
          const uint4 u = kt[e];
          kt[e] = (it.j0 + tile_row(e) >= it.klen) ? make_uint4(0u, 0u, 0u, 0u) : bf16x8_to_f16x8_scaled(u, ks);
        }
        fence_proxy_async_smem();
        mbar_arrive(bar(C::kBarK16));
        const float vs = exp2_int(cs.v);
#pragma unroll 2
        for (int i = 0; i < kVc; ++i) {
          const int e = ts + 256 * i;
          const uint4 u = vt[e];
          vt[e] = (it.j0 + tile_row(e) >= it.klen) ? make_uint4(0u, 0u, 0u, 0u) : bf16x8_to_f16x8_scaled(u, vs);
        }
        fence_proxy_async_smem();
        mbar_arrive(bar(C::kBarV16));
        sl2 = p.scale_log2 * exp2_int(-kexp - cs.q);
        cp = exp2_int(cs.g - cs.o - cs.v);
        dmul = exp2_int(cs.g);
        // Each warpgroup reads only its own 64 LSE/D entries, written by its
        // own threads tid < 64, so the two warpgroups never wait for each
        // other in the steps: a 128-thread named barrier publishes the
        // entries of step s before its passes, and a second one ends every
        // reader of step s before the entries of step s+1 overwrite them
        // (the previous item's last readers ended at its last step's second
        // barrier).
        if (tid < 64) {
          lse_s[64 * h + tid] = lse_next;
          dd_s[64 * h + tid] = d_next * dmul;
        }
        if (it.total > 1) load_row_terms(1, lse_next, d_next);
      }
      for (int s = 0; s < scs[5]; ++s) {
        const int gs = scs[7] + s;
        named_bar_sync(wg_bar, 128);
        do {
        if (!ok) break;
        const int q0 = (scs[2] + s % scs[3]) * kTileM;
        // Column c (query q0 + c) is visible iff this key row is inside
        // kv_len and, when causal, q0 + c >= j - offset.
        const int64_t cmin64 = p.mask.causal ? (static_cast<int64_t>(jrow) - scs[6] - q0) : INT64_MIN / 2;
        const int cmin = cmin64 > kTileM ? kTileM + 1 : (cmin64 < -1 ? -1 : static_cast<int>(cmin64));
        // Packed sequences: columns c >= cmax are query rows of the next
        // sequence; their weights and dS are set to 0 outright.  (In the padded
        // layout the rows past n_q read as zeros and carry LSE = -inf.)
        const int64_t cmax64 = static_cast<int64_t>(scs[1]) - q0;
        const int cmax = (!PACKED || cmax64 > kTileM) ? kTileM : static_cast<int>(cmax64);
        const bool need_mask =
            __any_sync(0xffffffffu, row_masked || cmin > 64 * h || (PACKED && cmax < 64 * h + 64));
        ok = wait_all(C::kBarSFull, static_cast<uint32_t>(gs & 1));
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
            uint32_t wq[8];
#pragma unroll
            for (int e = 0; e < 16; e += 2) {
              const int c = 64 * h + cq * 16 + e;
              const int r = (cq & 1) * 16 + e;
              const float s0 = __uint_as_float(cq < 2 ? sa[r] : sb[r]);
              const float s1 = __uint_as_float(cq < 2 ? sa[r + 1] : sb[r + 1]);
              float x0, x1;
              ffma2(x0, x1, s0, s1, sl2, sl2, nl[e], nl[e + 1]);
              if (need_mask) {
                x0 = (!row_masked && c >= cmin && (!PACKED || c < cmax)) ? x0 : -INFINITY;
                x1 = (!row_masked && c + 1 >= cmin && (!PACKED || c + 1 < cmax)) ? x1 : -INFINITY;
              }
              const float p0 = fast_exp2(x0), p1 = fast_exp2(x1);
              wq[e >> 1] = pack_f16x2(p0, p1);
              pf[cq * 16 + e] = p0;
              pf[cq * 16 + e + 1] = p1;
            }
            tmem_st8_nowait(tX + 64 * h + cq * 8, wq);
          }
          tmem_wait_st();
        }
        tc_fence_before_sync();
        mbar_arrive(bar(C::kBarPReady));
        ok = wait_all(C::kBarDPFull, static_cast<uint32_t>(gs & 1));
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
            uint32_t wq[8];
#pragma unroll
            for (int e = 0; e < 16; e += 2) {
              const int c = 64 * h + cq * 16 + e;
              const int r = (cq & 1) * 16 + e;
              const float g0 = __uint_as_float(cq < 2 ? da[r] : db[r]);
              const float g1 = __uint_as_float(cq < 2 ? da[r + 1] : db[r + 1]);
              float t0, t1, d0, d1;
              ffma2(t0, t1, g0, g1, cp, cp, nd[e], nd[e + 1]);
              fmul2(d0, d1, pf[cq * 16 + e], pf[cq * 16 + e + 1], t0, t1);
              if (need_mask) {
                d0 = (!row_masked && c >= cmin && (!PACKED || c < cmax)) ? d0 : 0.f;
                d1 = (!row_masked && c + 1 >= cmin && (!PACKED || c + 1 < cmax)) ? d1 : 0.f;
              }
              wq[e >> 1] = pack_f16x2(d0, d1);
            }
            // dS (queries contiguous per key row) for the dQ = dS K and
            // dK = dS^T Q products: this half's 64 queries fill one 128-byte
            // row of its block, the 16-byte chunk index XOR-swizzled with the
            // key row.
#pragma unroll
            for (int v = 0; v < 2; ++v) {
              const int chunk = cq * 2 + v;
              *reinterpret_cast<uint4*>(ds_row + ((chunk ^ (jj & 7)) * 16)) =
                  make_uint4(wq[4 * v], wq[4 * v + 1], wq[4 * v + 2], wq[4 * v + 3]);
            }
          }
        }
        fence_proxy_async_smem();
        tc_fence_before_sync();
        mbar_arrive(bar(C::kBarDSReady));
        } while (false);
        named_bar_sync(wg_bar, 128);
        const int nst = scs[5];
        if (ok && tid < 64 && s + 1 < nst) {
          lse_s[64 * h + tid] = lse_next;
          dd_s[64 * h + tid] = d_next * dmul;
        }
        if (ok && s + 2 < nst) slot_row_terms(s + 2, lse_next, d_next);
      }
      g += scs[5];
      ++ka;
    }
  } else if (warp >= 12) {
    // ============= dQ read-out, dK/dV epilogue (per item) ===============
    setmaxnreg_to<C::kRegsAux, C::kRegsLaunch>();
    const uint32_t quad = warp & 3;
    const int row = static_cast<int>(quad * 32 + lane);
    const uint32_t lane_base = (quad * 32u) << 16;
    const uint32_t tY = tmem + lane_base + C::kTY;
    bool ok = __all_sync(0xffffffffu, *abort_flag == 0);
    uint32_t rr[32];
    uint8_t* wstage = smem + C::kOffStage + quad * C::kDQWarpStage;
    volatile int* ro = reinterpret_cast<volatile int*>(smem + C::kOffRo + quad * 64);
    volatile float* rof = reinterpret_cast<volatile float*>(ro);
    // dQ read-out: each warp takes its 32 query rows of the tile (in Y) into
    // registers a 64-column round at a time and releases Y after the last
    // round's loads; it scales them back by 2^-(g + k) (dQ_acc = dS' K16,
    // CtaScale) and stages them as 32 x 32 fp32 boxes in the 128-byte swizzle
    // pattern (conflict-free stores), and one lane adds the boxes into the
    // fp32 accumulator with TMA reduce-add, a round at a time, the staging
    // memory being reused once a round's boxes have been read.  Rows past
    // n_q are clipped by the tensor map.
    auto stage_box = [&](uint8_t* dst_box, const uint32_t (&v)[32], float inv) {
      uint8_t* dst = dst_box + lane * 128;
#pragma unroll
      for (int c = 0; c < 8; ++c)
        *reinterpret_cast<float4*>(dst + ((c ^ (lane & 7)) * 16)) =
            make_float4(__uint_as_float(v[4 * c]) * inv, __uint_as_float(v[4 * c + 1]) * inv,
                        __uint_as_float(v[4 * c + 2]) * inv, __uint_as_float(v[4 * c + 3]) * inv);
    };
    // yz: the TMA coordinates of the warp's first row (worked out before the
    // step's wait, so no shared-memory read sits between the rounds), in:
    // whether that row is inside the sequence.
    auto reduce_round = [&](int first_box, TmaYZ yz, bool in) {
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0 && in) {
        // (Rows of the box past the sequence hold zeros: adding them is a
        // no-op on whatever rows lie there.)
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
    // The loop's counters (item k, items with steps ka, steps g) live in the
    // slot too.
    if (lane == 0) {
      ro[8] = 0;
      ro[9] = 0;
    }
    __syncwarp();
    for (int k = 0; ok; ++k) {
      int w = -1;
      if (!read_item(k, w)) break;
      float inv = 0.f;   // the dQ multiplier (read at the item's first dQ; the dK, dV ones go to the slot)
      if (bwd_item<SPLIT>(w, p).total > 0) {
        // Steps walk the query tiles [qt0, qt_end) of one head, then the
        // next; the item's fields live in this warp's slot.
        {
          const BwdItem it = bwd_item<SPLIT>(w, p);
          if (lane == 0) {
            ro[0] = it.b;
            ro[1] = static_cast<int>(it.nq_b);
            ro[2] = it.qt_first;
            ro[3] = it.qt_first + it.per_head;
            ro[4] = it.total;
            ro[5] = ro[8];
            ro[6] = w;
            ro[7] = it.head0;
          }
          __syncwarp();
        }
        int head = ro[7], qt = ro[2];
        for (int s = 0; s < ro[4] && ok; ++s) {
          const int gs = ro[5] + s;
          const int row0 = qt * kTileM + static_cast<int>(quad) * 32;
          const TmaYZ yz = q_tma(PACKED, p.lay, p.sh.Hq, ro[0], head, row0);
          const bool row_in = row0 < ro[1];
          ok = wait_all(C::kBarDQFull, static_cast<uint32_t>(gs & 1));
          if (!ok) break;
          tc_fence_after_sync();
          // The item's multipliers: published by the score warps before
          // their first dS of the item (whose barrier phase has completed
          // by now; it cannot run two phases ahead, since dS(g+1) follows
          // dP(g+1), which waits for this dQ's read-out).  The slot is
          // rewritten two items later, after the next item's first dP,
          // which waits for this item's last read-out.  (The K tile's
          // barrier could miss its phase instead: with one-step items it
          // may complete twice before these warps get there.)
          if (s == 0) {
            ok = wait_all(C::kBarDSReady, static_cast<uint32_t>(gs & 1));
            if (!ok) break;
            const float4 isc = iscale_s[ro[9] & 1];
            inv = isc.x;
            if (lane == 0) {
              rof[10] = isc.y;
              rof[11] = isc.z;
            }
          }
          // A round at a time: two 32-column loads behind one wait; Y is
          // handed back after the last round's loads.
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
            reduce_round(rd * C::kDQBoxesPerRound, yz, row_in);
          }
          __syncwarp();
          if (++qt == ro[3]) {
            qt = ro[2];
            ++head;
          }
        }
        if (!ok) break;
        ok = wait_all(C::kBarDKDV, static_cast<uint32_t>(ro[9] & 1));
        if (!ok) break;
        tc_fence_after_sync();
        w = ro[6];
      }
      __syncwarp();
      const float dk_scale = rof[10], dv_scale = rof[11];   // (unused by an item without steps)
      const BwdItem it = bwd_item<SPLIT>(opaque_int(w), p);   // (the loop's copy is dead)
      const int64_t j = it.j0 + row;
      const int64_t k_row_end = PACKED ? it.klen : p.sh.n_k;
      const bool in = j < k_row_end;
      int32_t kpos = 0;
      if constexpr (ROPE) kpos = in ? p.rot.pos[k_token(PACKED, p.lay, p.sh.n_k, it.b, j)] : 0;
      if constexpr (SPLIT) {
        // This item's share of dK, dV, in fp32, added into the split's sums
        // (dK turned back by the rotary first: the turn is linear).  The
        // tensor-memory loads are warp-collective: every lane takes part, and
        // only the rows inside the sequence are added.
        if (it.total > 0) {
          const int64_t arow = PACKED ? (static_cast<int64_t>(p.lay.cu_k[it.b]) + j) * p.sh.Hkv + it.hkv
                                      : (static_cast<int64_t>(it.b) * p.sh.Hkv + it.hkv) * p.sh.n_k + j;
#pragma unroll 1
          for (int cc = 0; cc < DH / 32; ++cc) {
            tmem_ld32(tmem + lane_base + C::kTdK + cc * 32, rr);
            float y[32];
#pragma unroll
            for (int e = 0; e < 32; ++e) y[e] = __uint_as_float(rr[e]) * dk_scale;
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
                  const int e = 8 * q4 + 2 * q;
                  rot_block(y[e], y[e + 1], cs4[q], sn4[q], y[e], y[e + 1]);
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
      } else {
        // dK, dV of the item's rows (zeros for an item without steps: its
        // keys are seen by no query, or lie past kv_len).
        uint4* dk = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.dK) +
                                             strided_off(PACKED, p.lay.sdk, p.sh.Hkv, p.lay.cu_k[it.b], it.b, it.hkv, j));
        uint4* dv = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.dV) +
                                             strided_off(PACKED, p.lay.sdv, p.sh.Hkv, p.lay.cu_k[it.b], it.b, it.hkv, j));
        // Rotary: the accumulated gradient is that of the rotated key; the
        // key's own gradient is it turned back by the key's angles (the
        // transpose of the rotation), formed here per 4-block chunk.
#pragma unroll 1
        for (int cc = 0; cc < DH / 32; ++cc) {
          uint32_t wq[16];
          if (it.total > 0) {
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
                  const int e = 8 * q4 + 2 * q;
                  float y0, y1;
                  rot_block(__uint_as_float(rr[e]) * dk_scale, __uint_as_float(rr[e + 1]) * dk_scale, cs4[q], sn4[q],
                            y0, y1);
                  wq[e >> 1] = pack_bf16x2(y0, y1);
                }
              }
            } else {
#pragma unroll
              for (int e = 0; e < 32; e += 2)
                wq[e >> 1] = pack_bf16x2(__uint_as_float(rr[e]) * dk_scale, __uint_as_float(rr[e + 1]) * dk_scale);
            }
          } else {
#pragma unroll
            for (int e = 0; e < 16; ++e) wq[e] = 0u;
          }
          if (in) {
#pragma unroll
            for (int v = 0; v < 4; ++v) dk[cc * 4 + v] = make_uint4(wq[4 * v], wq[4 * v + 1], wq[4 * v + 2], wq[4 * v + 3]);
          }
        }
#pragma unroll 1
        for (int cc = 0; cc < DV / 32; ++cc) {
          uint32_t wq[16];
          if (it.total > 0) {
            tmem_ld32(tmem + lane_base + C::kTdV + cc * 32, rr);
#pragma unroll
            for (int e = 0; e < 32; e += 2)
              wq[e >> 1] = pack_bf16x2(__uint_as_float(rr[e]) * dv_scale, __uint_as_float(rr[e + 1]) * dv_scale);
          } else {
#pragma unroll
            for (int e = 0; e < 16; ++e) wq[e] = 0u;
          }
          if (in) {
#pragma unroll
            for (int v = 0; v < 4; ++v) dv[cc * 4 + v] = make_uint4(wq[4 * v], wq[4 * v + 1], wq[4 * v + 2], wq[4 * v + 3]);
          }
        }
      }
      if (it.total > 0) {
        // The sums are in registers: the next item's first dK and dV
        // products may overwrite them.
        tc_fence_before_sync();
        mbar_arrive(bar(C::kBarAccFree));
        __syncwarp();
        if (lane == 0) {
          ro[8] = ro[8] + it.total;
          ro[9] = ro[9] + 1;
        }
        __syncwarp();
      }
    }
    if (lane == 0) bulk_wait_group0();
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, C::kTmemCols);
  }
  if (threadIdx.x == 0 && *abort_flag == 1) record_status(p.status, ATTN_ERR_TIMEOUT);
}

template <int DH, int DV>
cudaError_t launch_persistent_t(const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV,
                                const CUtensorMap& tmdO, const CUtensorMap& tmdQ, const BwdParams& p,
                                cudaStream_t stream) {
  using C = BwdPCfg<DH, DV>;
  // The split runs without a rotary only (the host never asks for both).
  auto kern = p.rot.pos ? (p.lay.packed ? attn_bwd_main_kernel<DH, DV, true, true, false>
                                        : attn_bwd_main_kernel<DH, DV, false, true, false>)
              : p.hsplit > 1 ? (p.lay.packed ? attn_bwd_main_kernel<DH, DV, true, false, true>
                                             : attn_bwd_main_kernel<DH, DV, false, false, true>)
                             : (p.lay.packed ? attn_bwd_main_kernel<DH, DV, true, false, false>
                                             : attn_bwd_main_kernel<DH, DV, false, false, false>);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (e != cudaSuccess) return e;
  kern<<<static_cast<unsigned>(p.ctas), C::kThreads, C::kSmemBytes, stream>>>(tmQ, tmK, tmV, tmdO, tmdQ, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attn_bwd_main_persistent(int dh, int dv, const CUtensorMap& tmQ, const CUtensorMap& tmK,
                                            const CUtensorMap& tmV, const CUtensorMap& tmdO,
                                            const CUtensorMap& tmdQ, const BwdParams& p, cudaStream_t stream) {
  if (dh == 128 && dv == 128) return launch_persistent_t<128, 128>(tmQ, tmK, tmV, tmdO, tmdQ, p, stream);
  if (dh == 64 && dv == 64) return launch_persistent_t<64, 64>(tmQ, tmK, tmV, tmdO, tmdQ, p, stream);
  if (dh == 128 && dv == 64) return launch_persistent_t<128, 64>(tmQ, tmK, tmV, tmdO, tmdQ, p, stream);
  return cudaErrorInvalidValue;
}

}  // namespace esd
