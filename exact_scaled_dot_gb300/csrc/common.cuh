// common.cuh -- launch parameters and the visible-set closed forms shared by
// the host code and the kernels.
//
// Visible set ("Appendix A.10 -- Attention matrices and backpropagation",
// eq. A.10.1 and section A.10.6; "Chapter 31 -- attention backprop",
// section 1 for n_q != n_k): key j is visible to query row i of batch b iff
//     j < kv_len[b]   and, when causal,   j <= i + offset(b),
// for the rows i < q_len(b) that exist.  offset(b) is one offset for the
// whole batch, or, for packed variable-length sequences, kv_len[b] - q_len[b]
// (each sequence's last query aligned with its last key).  Both conditions
// are upper bounds on j, so each row has a single key limit
//     lim(b, i) = min(kv_len[b], causal ? i + offset(b) + 1 : n_k)
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
  int32_t has_q_len;               // rows i >= q_len[b] do not exist (packed sequences)
  int32_t offset_from_lengths;     // causal offset(b) = kv_len[b] - q_len[b]
  int32_t q_len[ATTN_MAX_BATCH];   // valid when has_q_len
};

struct ShapeParams {
  int32_t B, Hq, Hkv, n_q, n_k, group;  // group = Hq / Hkv
};

__host__ __device__ __forceinline__ int64_t key_len(const MaskParams& m, int n_k, int b) {
  return m.has_kv_len ? static_cast<int64_t>(m.kv_len[b]) : static_cast<int64_t>(n_k);
}

// Query rows of batch element b (n_q unless the rows are per-sequence).
__host__ __device__ __forceinline__ int64_t query_len(const MaskParams& m, int n_q, int b) {
  return m.has_q_len ? static_cast<int64_t>(m.q_len[b]) : static_cast<int64_t>(n_q);
}

__host__ __device__ __forceinline__ int64_t causal_offset(const MaskParams& m, int b) {
  return m.offset_from_lengths ? static_cast<int64_t>(m.kv_len[b]) - m.q_len[b] : m.offset;
}

// lim(b, i): keys j < lim are visible to row i.
__host__ __device__ __forceinline__ int64_t row_key_limit(const MaskParams& m, int n_k, int b,
                                                          int64_t i) {
  int64_t lim = key_len(m, n_k, b);
  if (m.causal) {
    const int64_t c = i + causal_offset(m, b) + 1;
    lim = c < lim ? c : lim;
  }
  return lim;
}

// Number of key tiles a query tile [i0, i0 + kTileM) must visit: every tile
// below the last row's limit is non-empty, every tile above is empty.
__host__ __device__ __forceinline__ int kv_tiles_for_q_tile(const MaskParams& m, int n_q, int n_k,
                                                            int b, int64_t i0) {
  const int64_t nq_b = query_len(m, n_q, b);
  if (i0 >= nq_b) return 0;
  int64_t i_last = i0 + kTileM - 1;
  if (i_last > nq_b - 1) i_last = nq_b - 1;
  const int64_t lim = row_key_limit(m, n_k, b, i_last);
  if (lim <= 0) return 0;
  return static_cast<int>((lim + kTileN - 1) / kTileN);
}

// Rows [r0, r1) of key tile j (tile-relative) lie in [kv_len, row_end):
// rows that hold caller memory but no visible key (row_end = n_k for the
// padded layout; for packed sequences the tile's rows past the sequence
// belong to the next one, row_end = INT32_MAX).  False when there are none.
__host__ __device__ __forceinline__ bool padded_rows(const MaskParams& m, int row_end, int b, int j, int& r0,
                                                     int& r1) {
  const int64_t j0 = static_cast<int64_t>(j) * kTileN;
  int64_t lo = key_len(m, row_end, b) - j0, hi = static_cast<int64_t>(row_end) - j0;
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
  const int64_t nq_b = query_len(m, n_q, b);
  if (j0 >= key_len(m, n_k, b)) return nq_b;
  if (!m.causal) return 0;
  int64_t i = j0 - causal_offset(m, b);
  if (i < 0) i = 0;
  return i < nq_b ? i : nq_b;
}

// Where the rows of a tensor live.  Padded layout: [B][H][n][d], row i of
// (b, h) at (b H + h) n + i.  Packed variable-length sequences: [T][H][d]
// with the tokens of sequence b at cu[b] .. cu[b+1] - 1, row i of (b, h) at
// (cu[b] + i) H + h.  The backward's fp16 copy of Q and its fp32 dQ
// accumulator follow the layout of Q; LSE and D are [B][H][n] (padded) or
// [H][T] (packed).
// Element strides of one user tensor (its innermost index, d, has stride 1):
// `row` between consecutive rows of a head (tokens in the packed layout),
// `head` between consecutive heads; in the padded layout the batch stride is
// H head.  The workspace copies (fp16 Q and dO, the dQ accumulator) always use
// the contiguous strides of the layout.
struct TensorStrides {
  int64_t row, head;
};

struct LayoutParams {
  int32_t packed;
  int32_t cu_q[ATTN_MAX_BATCH + 1];   // packed: first query token of sequence b
  int32_t cu_k[ATTN_MAX_BATCH + 1];   // packed: first key token of sequence b
  int64_t total_q;                    // packed: query tokens
  // User tensors: Q, K, V, O (and O_lo), dO, dQ, dK, dV.
  TensorStrides sq, sk, sv, so, sdo, sdq, sdk, sdv;
};

// Element offset of row i of (b, h) in a user tensor with strides `s` and H
// heads (cu: the packed layout's first token of sequence b).
__host__ __device__ __forceinline__ int64_t strided_off(bool packed, const TensorStrides& s, int H, int32_t cu, int b,
                                                        int h, int64_t i) {
  return packed ? (static_cast<int64_t>(cu) + i) * s.row + static_cast<int64_t>(h) * s.head
                : (static_cast<int64_t>(b) * H + h) * s.head + i * s.row;
}

// The helpers take the layout kind as their first argument: the kernels are
// compiled once per kind and pass it as a constant, so the padded layout's
// index arithmetic carries no trace of the packed one.
// Element row (in units of the row width) of query row i of (b, h).
__host__ __device__ __forceinline__ int64_t q_row(bool packed, const LayoutParams& L, int Hq, int n_q, int b, int h,
                                                  int64_t i) {
  return packed ? (static_cast<int64_t>(L.cu_q[b]) + i) * Hq + h : (static_cast<int64_t>(b) * Hq + h) * n_q + i;
}
__host__ __device__ __forceinline__ int64_t k_row(bool packed, const LayoutParams& L, int Hkv, int n_k, int b, int h,
                                                  int64_t j) {
  return packed ? (static_cast<int64_t>(L.cu_k[b]) + j) * Hkv + h : (static_cast<int64_t>(b) * Hkv + h) * n_k + j;
}
// Index of the LSE / D entry of query row i of (b, h).
__host__ __device__ __forceinline__ int64_t q_vec(bool packed, const LayoutParams& L, int Hq, int n_q, int b, int h,
                                                  int64_t i) {
  return packed ? static_cast<int64_t>(h) * L.total_q + L.cu_q[b] + i : (static_cast<int64_t>(b) * Hq + h) * n_q + i;
}
// TMA coordinates (y, z) of row i of (b, h) in the 3-D view of a tensor:
// padded views are [B H][n][d] (y = row, z = b H + h), packed views
// [T][H][d] (y = head, z = token).
struct TmaYZ {
  int32_t y, z;
};
__device__ __forceinline__ TmaYZ q_tma(bool packed, const LayoutParams& L, int Hq, int b, int h, int i) {
  return packed ? TmaYZ{h, L.cu_q[b] + i} : TmaYZ{i, b * Hq + h};
}
__device__ __forceinline__ TmaYZ k_tma(bool packed, const LayoutParams& L, int Hkv, int b, int h, int j) {
  return packed ? TmaYZ{h, L.cu_k[b] + j} : TmaYZ{j, b * Hkv + h};
}

// Token of query row i / key row j of batch element b: the row of its
// positions and of its cos/sin table (padded b n + i, packed cu[b] + i).
__host__ __device__ __forceinline__ int64_t q_token(bool packed, const LayoutParams& L, int n_q, int b, int64_t i) {
  return packed ? static_cast<int64_t>(L.cu_q[b]) + i : static_cast<int64_t>(b) * n_q + i;
}
__host__ __device__ __forceinline__ int64_t k_token(bool packed, const LayoutParams& L, int n_k, int b, int64_t j) {
  return packed ? static_cast<int64_t>(L.cu_k[b]) + j : static_cast<int64_t>(b) * n_k + j;
}

// Rotary embedding: the positions of the rows a kernel turns and the
// frequencies w_k = base^(-2k/d), k < d/2, as fp32 pairs w_hi + w_lo (w_lo
// the rounding residual of w_hi, so that the rounding of w does not grow
// with the position).  pos == nullptr: no rotation.
struct RotaryAngles {
  const int32_t* pos;
  float w_hi[64];
  float w_lo[64];
};

// Rotated copies ahead of the attention kernels, over two segments (the
// query and the key tokens): each writes its tokens' rows rotated, read from
// the caller's strided tensor X and written contiguous in X's layout (padded
// [B H][n][d], packed [T][H][d]).
struct RopeSegment {
  int64_t tokens;              // padded: B n; packed: T (0: empty segment)
  int32_t n;                   // padded: rows per (b, h)
  int32_t H;                   // heads of X
  const int32_t* pos;          // [tokens]
  const void* X;               // bf16 rows to rotate (strides sx)
  TensorStrides sx;
  void* Y;                     // rotated rows, contiguous
};
struct RopePrepParams {
  int32_t d, packed;
  RopeSegment seg[2];
  float w_hi[64];              // as in RotaryAngles
  float w_lo[64];
};

struct FwdParams {
  ShapeParams sh;
  MaskParams mask;
  LayoutParams lay;
  float scale_log2;            // scale * log2(e)
  uint64_t wait_limit_ns;
  void* O;                     // bf16 [B][Hq][n_q][d_v]
  void* O_lo;                  // bf16 rounding residual of O, or nullptr
  float* LSE;                  // fp32 [B][Hq][n_q]
  const int32_t* vexp;         // [B Hkv][nkt] exponents of the fp16 V tiles (attn_v16_kernel)
  int32_t nkt;                 // key tiles per head of the fp16 V buffer
  unsigned int* status;        // device status word
};


// The forward's fp16 copy of V: tile j of (b, h) re-encoded as V 2^vexp
// (f16range.cuh), rows past the key length zero, in a [B Hkv][nkt 128][d_v]
// buffer in both layouts.
struct V16Params {
  ShapeParams sh;
  MaskParams mask;
  LayoutParams lay;
  int32_t nkt;
  const void* V;               // bf16, the caller's layout
  void* V16;                   // fp16 [B Hkv][nkt 128][d_v]
  int32_t* vexp;               // [B Hkv][nkt]; tiles past the key length are not written
  unsigned int* status;
  // Rotary: prep_rows extra rows of blocks in the same launch work through
  // rp (the rotated queries and keys); 0 without a rotary.
  int32_t prep_rows;
  RopePrepParams rp;
};

struct BwdParams {
  ShapeParams sh;
  MaskParams mask;
  LayoutParams lay;
  float scale;                 // raw scale (dK epilogue)
  float scale_log2;            // scale * log2(e)
  uint64_t wait_limit_ns;
  const float* LSE;            // fp32 [B][Hq][n_q]
  const float* D;              // fp32 [B][Hq][n_q]
  const float4* tilemax;       // per 128-row query tile: (max ||dO_i||, max |D_i|, e_Q, e_dO), [B Hq][nqt]
  int32_t nqt;                 // query tiles per head (of the longest sequence)
  const float2* grpexp;        // [B Hkv]: the exponents of the group's fp16 Q and dO tiles
  float* dQacc;                // fp32 [B][Hq][n_q][d_h]
  void* dK;                    // bf16 [B][Hkv][n_k][d_h]
  void* dV;                    // bf16 [B][Hkv][n_k][d_v]
  unsigned int* status;
  RotaryAngles rot;            // rotary: the keys' positions (dK turned back in the epilogue)
  // Query-head split: blockIdx.z of hsplit takes group / hsplit of the KV
  // head's query heads; with hsplit > 1 every CTA adds its fp32 share of dK,
  // dV into dKacc, dVacc (rows [tokens_k Hkv][d], zeroed beforehand) instead
  // of writing dK, dV.
  int32_t hsplit;
  float* dKacc;
  float* dVacc;
  // Schedule: persistent = 0, one CTA per work item (grid B Hkv x key tiles
  // x hsplit); persistent = 1, ctas CTAs take the nitems work items (B Hkv
  // key tiles, times hsplit), the first ctas by block index, the rest from
  // *work_ctr (zeroed by the backward's first stage).
  int32_t persistent;
  unsigned int* work_ctr;
  int32_t nitems;
  int32_t ctas;
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
  int16_t batch_order[ATTN_MAX_BATCH];  // batches by descending key range: CTA dispatch order
};

// The projection products (A.10.10-A.10.11): C = sum_s A_s B_s, row-major
// bf16 operands through TMA maps, C row-major with leading dimension ldc.
enum GemmKind : int {
  kGemmXW = 0,    // Y = X W:     A [M][K] K-major, B [K][N] MN-major, C bf16
  kGemmXtG = 1,   // dW = X^T G:  A [K][M] MN-major, B [K][N] MN-major, C fp32
  kGemmGWt = 2,   // dX = G W^T:  A [M][K] K-major, B [N][K] K-major, C bf16 (up to 3 sources)
};
struct GemmParams {
  int64_t M;                   // output rows
  int32_t N;                   // output columns
  int32_t nsrc;                // products summed (1..3)
  int32_t K[3];                // contraction length of each product
  int32_t ldc;
  void* C;
  uint64_t wait_limit_ns;
  unsigned int* status;
};

// Default limit of every bounded wait inside the kernels.
constexpr uint64_t kDefaultWaitLimitNs = 2000000000ull;  // 2 s

// Kernel launchers (defined next to their kernels).
cudaError_t launch_attn_fwd(int dh, int dv, const CUtensorMap& tmQ, const CUtensorMap& tmK,
                            const CUtensorMap& tmV, const FwdParams& p, cudaStream_t stream);
cudaError_t launch_attn_v16(int dv, const V16Params& p, cudaStream_t stream);
cudaError_t launch_attn_decode(int dh, int dv, const CUtensorMap& tmK, const CUtensorMap& tmV, const DecParams& p,
                               cudaStream_t stream);
cudaError_t launch_attn_bwd_main(int dh, int dv, const CUtensorMap& tmQ, const CUtensorMap& tmK,
                                 const CUtensorMap& tmV, const CUtensorMap& tmdO, const CUtensorMap& tmdQ,
                                 const BwdParams& p, cudaStream_t stream);
// The persistent schedule's kernels (attn_bwd_persist.cu); launch_attn_bwd_main
// dispatches to it when p.persistent is set.
cudaError_t launch_attn_bwd_main_persistent(int dh, int dv, const CUtensorMap& tmQ, const CUtensorMap& tmK,
                                            const CUtensorMap& tmV, const CUtensorMap& tmdO,
                                            const CUtensorMap& tmdQ, const BwdParams& p, cudaStream_t stream);
// rot_q: the queries' positions (rotary: Q is rotated as it is read), or nullptr.
// work_ctr: the main kernel's work counter, zeroed by this stage.
cudaError_t launch_attn_bwd_preprocess(const ShapeParams& sh, const LayoutParams& lay, int dv, int dh,
                                       const void* Q, const void* O, const void* O_lo, const void* dO, float* D,
                                       float4* tilemax, float2* grpexp, unsigned int* work_ctr, float* dQacc,
                                       void* Q16, void* dO16, const RotaryAngles* rot_q, unsigned int* status,
                                       cudaStream_t stream);
cudaError_t launch_proj_gemm(int kind, const CUtensorMap* tA, const CUtensorMap* tB, const GemmParams& p,
                             cudaStream_t stream);
cudaError_t launch_rope_prep(const RopePrepParams& p, cudaStream_t stream);
// heads_b = 0: one tensor (xb, yb unused).
cudaError_t launch_rope(int64_t tokens, int d, int heads_a, int heads_b, const int32_t* pos, const float* w_hi,
                        const float* w_lo, int inverse, const void* xa, void* ya, const void* xb, void* yb, cudaStream_t stream);
// Zero n floats (n a multiple of 4, 16-byte aligned).
cudaError_t launch_zero_f32(float* p, int64_t n, cudaStream_t stream);
// dK, dV (bf16, caller strides) from the fp32 sums of a query-head split:
// rows of (b, h) in the accumulators are [tokens_k Hkv][d] (padded token
// b n_k + j, row (b Hkv + h) n_k + j; packed row token Hkv + h).
cudaError_t launch_attn_bwd_kv_finalize(const ShapeParams& sh, const LayoutParams& lay, int64_t tokens_k, int dh,
                                        int dv, const float* dKacc, const float* dVacc, void* dK, void* dV,
                                        cudaStream_t stream);
// dQ = scale * accumulator (elems elements of rows of dh); contiguous dQ, or
// row r at (r / n_inner) s_outer + (r % n_inner) s_inner.  With rot_q (the
// queries' positions) each row is turned back by its token's angles: the
// token of row r is r / n_inner when packed (rows are tokens of Hq heads),
// else (r / n_inner / Hq) n_inner + r % n_inner (rows are heads of n_q rows).
cudaError_t launch_attn_bwd_finalize(int64_t elems, int dh, int n_inner, int64_t s_outer, int64_t s_inner,
                                     bool contiguous, float scale, const float* dQacc, void* dQ,
                                     const RotaryAngles* rot_q, bool packed, int Hq, cudaStream_t stream);

}  // namespace esd
