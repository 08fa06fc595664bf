// common.cuh -- launch parameters and the visible-set closed forms shared by
// the host code and the kernels.
//
// Visible set ("Appendix A.10 -- Attention matrices and backpropagation",
// eq. A.10.1 and section A.10.6; "Chapter 31 -- attention backprop",
// section 1 for n_q != n_k): key j is visible to query row i of batch b iff
//     j < kv_len[b]   and, when causal,   j <= i + offset.
// Both conditions are upper bounds on j, so each row has a single key limit
//     lim(b, i) = min(kv_len[b], causal ? i + offset + 1 : n_k)
// and j is visible iff j < lim(b, i).  lim is non-decreasing in i, which
// makes whole-tile classification a pair of comparisons.
#pragma once

#include <cstdint>
#include <cuda.h>

#include "../../include/attn.h"

namespace esd {

constexpr int kTileM = 128;  // query rows per tile
constexpr int kTileN = 128;  // key rows per tile
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

struct MaskParams {
  int32_t causal;
  int32_t has_kv_len;
  int64_t offset;                  // effective causal offset, clamped to [0, n_k]
  int32_t kv_len[ATTN_MAX_BATCH];  // valid when has_kv_len
};

struct ShapeParams {
  int32_t B, Hq, Hkv, n_q, n_k, group;  // group = Hq / Hkv
};

__host__ __device__ __forceinline__ int64_t key_len(const MaskParams& m, int n_k, int b) {
  return m.has_kv_len ? static_cast<int64_t>(m.kv_len[b]) : static_cast<int64_t>(n_k);
}

// lim(b, i): keys j < lim are visible to row i.
__host__ __device__ __forceinline__ int64_t row_key_limit(const MaskParams& m, int n_k, int b,
                                                          int64_t i) {
  int64_t lim = key_len(m, n_k, b);
  if (m.causal) {
    const int64_t c = i + m.offset + 1;
    lim = c < lim ? c : lim;
  }
  return lim;
}

// Number of key tiles a query tile [i0, i0 + kTileM) must visit: every tile
// below the last row's limit is non-empty, every tile above is empty.
__host__ __device__ __forceinline__ int kv_tiles_for_q_tile(const MaskParams& m, int n_q, int n_k,
                                                            int b, int64_t i0) {
  if (i0 >= n_q) return 0;
  int64_t i_last = i0 + kTileM - 1;
  if (i_last > n_q - 1) i_last = n_q - 1;
  const int64_t lim = row_key_limit(m, n_k, b, i_last);
  if (lim <= 0) return 0;
  return static_cast<int>((lim + kTileN - 1) / kTileN);
}

// Rows [r0, r1) of key tile j (tile-relative) lie in [kv_len, n_k): rows
// that hold caller memory but no visible key.  False when there are none.
__host__ __device__ __forceinline__ bool padded_rows(const MaskParams& m, int n_k, int b, int j, int& r0,
                                                     int& r1) {
  const int64_t j0 = static_cast<int64_t>(j) * kTileN;
  int64_t lo = key_len(m, n_k, b) - j0, hi = static_cast<int64_t>(n_k) - j0;
  if (lo < 0) lo = 0;
  if (hi > kTileN) hi = kTileN;
  if (lo >= hi) return false;
  r0 = static_cast<int>(lo);
  r1 = static_cast<int>(hi);
  return true;
}

// First query row that sees key j0 (the smallest i with lim(i) > j0), or
// n_q when no row does.
__host__ __device__ __forceinline__ int64_t first_row_seeing_key(const MaskParams& m, int n_q,
                                                                 int n_k, int b, int64_t j0) {
  if (j0 >= key_len(m, n_k, b)) return n_q;
  if (!m.causal) return 0;
  int64_t i = j0 - m.offset;
  if (i < 0) i = 0;
  return i < n_q ? i : n_q;
}

struct FwdParams {
  ShapeParams sh;
  MaskParams mask;
  float scale_log2;            // scale * log2(e)
  uint64_t wait_limit_ns;
  void* O;                     // bf16 [B][Hq][n_q][d_v]
  void* O_lo;                  // bf16 rounding residual of O, or nullptr
  float* LSE;                  // fp32 [B][Hq][n_q]
  unsigned int* status;        // device status word
};

struct BwdParams {
  ShapeParams sh;
  MaskParams mask;
  float scale;                 // raw scale (dK epilogue)
  float scale_log2;            // scale * log2(e)
  uint64_t wait_limit_ns;
  const float* LSE;            // fp32 [B][Hq][n_q]
  const float* D;              // fp32 [B][Hq][n_q]
  const float2* tilemax;       // per 128-row query tile: (max ||dO_i||, max |D_i|)
  int32_t nqt;                 // query tiles per head
  float* dQacc;                // fp32 [B][Hq][n_q][d_h]
  void* dK;                    // bf16 [B][Hkv][n_k][d_h]
  void* dV;                    // bf16 [B][Hkv][n_k][d_v]
  unsigned int* status;
};

struct DecParams {
  ShapeParams sh;
  MaskParams mask;
  float scale_log2;            // scale * log2(e)
  uint64_t wait_limit_ns;
  const void* Q;               // bf16 [B][Hq][n_q][d_h], gathered by threads
  void* O;                     // bf16 [B][Hq][n_q][d_v]
  void* O_lo;                  // bf16 rounding residual of O, or nullptr
  float* LSE;                  // fp32 [B][Hq][n_q]
  float* Opart;                // fp32 [nsplit][B*Hq*n_q][d_v] range partials (nsplit > 1)
  float* Lpart;                // fp32 [nsplit][B*Hq*n_q] range log-sum-exps (nsplit > 1)
  int32_t heads_per_tile;      // query heads packed into one 128-row tile
  int32_t chunks;              // row tiles per KV head
  int32_t nsplit;              // key ranges per row tile
  unsigned int* status;
};

// Default limit of every bounded wait inside the kernels.
constexpr uint64_t kDefaultWaitLimitNs = 2000000000ull;  // 2 s

// Kernel launchers (defined next to their kernels).
cudaError_t launch_attn_fwd(int dh, int dv, const CUtensorMap& tmQ, const CUtensorMap& tmK,
                            const CUtensorMap& tmV, const FwdParams& p, cudaStream_t stream);
cudaError_t launch_attn_decode(int dh, int dv, const CUtensorMap& tmK, const CUtensorMap& tmV, const DecParams& p,
                               cudaStream_t stream);
cudaError_t launch_attn_bwd_main(int dh, int dv, const CUtensorMap& tmQ, const CUtensorMap& tmK,
                                 const CUtensorMap& tmV, const CUtensorMap& tmdO, const CUtensorMap& tmdQ,
                                 const BwdParams& p, cudaStream_t stream);
cudaError_t launch_attn_bwd_preprocess(int64_t bhq, int n_q, int dv, int dh, const void* Q, const void* O,
                                       const void* O_lo, const void* dO, float* D, float2* tilemax, float* dQacc,
                                       void* Q16, cudaStream_t stream);
cudaError_t launch_attn_bwd_finalize(int64_t elems, float scale, const float* dQacc, void* dQ,
                                     cudaStream_t stream);

}  // namespace esd
