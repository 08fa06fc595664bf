/*
 * attn.h -- C ABI of the GB300 (sm_103a) masked scaled dot-product attention
 * library, forward and backward.
 *
 * What is computed.  For every batch element b and query head r, with KV head
 * h = g(r) = floor(r / (Hq / Hkv)) ("Appendix A.10 -- Attention matrices and
 * backpropagation", section A.10.5: MHA when Hkv = Hq, MQA when Hkv = 1, GQA
 * in between):
 *   S_ij = scale * q_i . k_j              for j in the visible set V_i   (A.10.1)
 *   A_ij = exp(S_ij - m_i) / sum_{r in V_i} exp(S_ir - m_i),
 *          m_i = max_{j in V_i} S_ij, and A_ij = 0 off V_i               (A.10.2)
 *   O    = A V                                                           (A.10.3)
 *   LSE_i = m_i + ln sum_{j in V_i} exp(S_ij - m_i)
 * and the backward pass, given dO = dL/dO:
 *   dV   = A^T dO                                                        (A.10.5)
 *   dA   = dO V^T                                                        (A.10.6)
 *   dS_ij = A_ij (dA_ij - c_i) on V_i, 0 elsewhere,
 *          c_i = sum_j A_ij dA_ij = sum_l dO_il O_il                     (A.10.7)
 *   dQ   = scale * dS K,     dK = scale * dS^T Q                         (A.10.8-9)
 * with dK, dV summed over the query heads that share a KV head (A.10.5).
 * The usual scale is 1/sqrt(d_h); it is passed explicitly.
 *
 * Visible set.  V_i = { j : j < kv_len[b], and j <= i + causal_offset when
 * causal }.  Causal self-attention is V_i = { j <= i } ("Appendix A.10",
 * section A.10.6); for n_q != n_k the default offset n_k - n_q aligns the
 * last query with the last key (a new chunk of queries over a long history,
 * "Chapter 31 -- attention backprop", section 1).  kv_len is key padding.
 * A row with an empty visible set is undefined (A.10.2) and rejected
 * ("Chapter 31", section 3): every call checks this in closed form on the
 * host and returns ATTN_ERR_EMPTY_ROW before launching anything.
 *
 * Layout.  Tensors are row-major with the innermost index last:
 *   Q, dQ   [B][Hq ][n_q][d_h]  bf16        K, dK [B][Hkv][n_k][d_h] bf16
 *   O, dO   [B][Hq ][n_q][d_v]  bf16        V, dV [B][Hkv][n_k][d_v] bf16
 *   LSE, D  [B][Hq ][n_q]       fp32
 * (the packed variable-length entry points below use token-major tensors).
 * They are contiguous unless the call's attn_strides say otherwise (below);
 * LSE is always contiguous.  Supported head widths (d_h, d_v): (64, 64),
 * (128, 128), (128, 64).  Every tensor pointer must be 16-byte aligned.
 *
 * Ownership and execution.  The caller allocates and owns every buffer,
 * including the forward and backward workspaces; the library allocates no
 * device memory.  It keeps a little state between calls: a cached driver
 * entry point and, per device, the device addresses of its status word and
 * of attn_bwd_noalloc's static buffer, looked up on the first call there.
 * Those addresses belong to the device's primary context: after
 * cudaDeviceReset (or anything else that destroys and recreates that
 * context) the library must not be called on that device again in the same
 * process.  Device pointers refer to memory of the current CUDA device.  `stream` is a
 * cudaStream_t (NULL = the legacy default stream); every call only enqueues
 * work on it and returns without synchronising.  Host arrays (kv_len) are
 * read during the call only.
 *
 * Errors.  Every function returns ATTN_OK (0) or one of the codes below; no
 * exception or abort crosses the ABI.  Argument checks happen before any
 * CUDA call.  Device-side conditions are recorded in a device status word
 * that attn_get_status() reads and attn_clear_status() resets:
 * ATTN_ERR_TIMEOUT (a bounded wait ran out; while it is set, the kernels
 * return immediately without writing outputs) or ATTN_ERR_RANGE (an input
 * tile was too large for the fp16 operands, below; the outputs of that call
 * are not to be trusted, later calls run normally).
 *
 * Precision.  Inputs and outputs are bf16 with fp32 accumulation.  Q K^T in
 * the forward runs on bf16 operands; P V and every backward product run on
 * fp16 operands (11 significant bits, so that the weights and dS keep more
 * precision than bf16 gives them).  Each fp16 operand is the bf16 input
 * times a power of two 2^e chosen from the largest magnitude M it holds, so
 * that 2^11 <= M 2^e < 2^15 (e a multiple of 4), and the products are
 * unscaled exactly.  The unit that shares one e is a 128-key tile of V in
 * the forward, a 128-key tile of K and of V in the backward, and all query
 * rows of Q (and of dO) that share a KV head in the backward.  The
 * re-encoding is therefore exact at any input scale: every value down to
 * about 2^-28 M is kept, for any M below 2^46; a tile with M >= 2^46
 * saturates and sets ATTN_ERR_RANGE.  (e is clamped to [-30, 30]: a unit
 * whose M is below 2^-16 still keeps every value down to 2^-47.)
 */
#ifndef EXACT_SCALED_DOT_GB300_ATTN_H
#define EXACT_SCALED_DOT_GB300_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define ATTN_ABI_VERSION 12

/* Status codes. */
#define ATTN_OK               0
#define ATTN_ERR_NULL         1  /* a required pointer is NULL                         */
#define ATTN_ERR_SHAPE        2  /* non-positive size, Hq % Hkv != 0, kv_len out of   */
                                 /* [1, n_k], B > ATTN_MAX_BATCH, n_q or n_k above       */
                                 /* 65535*128, size overflow                            */
#define ATTN_ERR_UNSUPPORTED  3  /* (d_h, d_v) not one of the supported pairs          */
#define ATTN_ERR_ALIGN        4  /* a tensor pointer is not 16-byte aligned            */
#define ATTN_ERR_EMPTY_ROW    5  /* some query row has an empty visible set            */
#define ATTN_ERR_SCALE        6  /* scale is not finite or not > 0                     */
#define ATTN_ERR_WORKSPACE    7  /* workspace NULL, misaligned or too small            */
#define ATTN_ERR_CUDA         8  /* a CUDA runtime/driver call or launch failed        */
#define ATTN_ERR_TIMEOUT      9  /* a kernel's bounded wait ran out (device status)    */
#define ATTN_ERR_DEVICE      10  /* the current device is not an sm_103 GPU            */
#define ATTN_ERR_RANGE       11  /* an input tile held a magnitude of 2^46 or more,    */
                                 /* beyond the scaled fp16 operands (device status)    */

/* Largest batch whose per-batch key lengths travel with the launch. */
#define ATTN_MAX_BATCH 512

/* Sentinel for attn_mask.causal_offset: use n_k - n_q. */
#define ATTN_OFFSET_DEFAULT INT64_MIN

typedef struct {
  int32_t B;    /* batch                                     */
  int32_t Hq;   /* query heads                               */
  int32_t Hkv;  /* key/value heads; Hq % Hkv == 0            */
  int32_t n_q;  /* query rows per head                       */
  int32_t n_k;  /* key rows per head                         */
  int32_t d_h;  /* query/key width                           */
  int32_t d_v;  /* value width                               */
} attn_shape;

typedef struct {
  int32_t causal;          /* 0: no causal bound; 1: j <= i + causal_offset          */
  int32_t reserved;        /* must be 0                                               */
  int64_t causal_offset;   /* ATTN_OFFSET_DEFAULT, or an explicit offset (>= 0 keeps  */
                           /* row 0 non-empty)                                        */
  const int32_t* kv_len;   /* NULL (= n_k for all) or HOST array [B], each in [1,n_k] */
} attn_mask;


/* Element strides of one tensor whose innermost index (d) is contiguous:
 * `row` = elements between consecutive rows of one head (between
 * consecutive tokens in the packed layout), `head` = elements between
 * consecutive heads.  In the padded layout [B][H][n][d] the batch stride is
 * H * head: a tensor sliced along d, or with padded rows or heads, fits; a
 * sequence-major [B][n][H][d] tensor does not and goes through the packed
 * entry points (one sequence per batch element).  Both strides must be
 * multiples of 8 (16-byte rows; ATTN_ERR_ALIGN otherwise) and at least d
 * (ATTN_ERR_SHAPE).  {0, 0} means the contiguous strides of the layout. */
typedef struct {
  int64_t row, head;
} attn_tensor_strides;

/* Strides of a call's tensors ("Appendix A.10", section A.10.5: the
 * B x H x n x d tensors and their head concatenation); NULL = every tensor
 * contiguous.  O_lo has O's strides.  Every entry is checked, also those of
 * tensors the call does not take ({0, 0} passes).  A Q, K or V that is a
 * slice of one fused projection output [T][(Hq + 2 Hkv) d] (token stride
 * (Hq + 2 Hkv) d, head stride d) is read in place by the packed entry
 * points, and dQ, dK, dV may be written into the matching slices of one
 * fused gradient buffer.  Output views must not overlap one another or an
 * input; nothing outside a view is written. */
typedef struct {
  attn_tensor_strides q, k, v, o, dO, dq, dk, dv;
} attn_strides;

/* Rotary position embedding fused into the attention entry points
 * ("Chapter 15 -- matrix formulas", section 15.6: the scores are those of
 * the rotated rows q~_i = R_i q_i, k~_j = R_j k_j; "Chapter 31 -- attention
 * backprop", section 5: the gradients of q and k are those of q~ and k~
 * turned back by the opposite angles).  NULL = no rotation.  The rotation is
 * attn_rope's (same angles, same bf16 rounding of each rotated row), over
 * the whole width d_h of Q and K; V is not rotated.  The forward with a
 * rotary equals, bit for bit, attn_rope on Q and K followed by the forward
 * without one.  The backward takes the un-rotated Q and K and returns the
 * gradients of the un-rotated Q and K; their turn back happens in fp32,
 * before the one rounding to bf16.
 * pos_q, pos_k: device int32 positions of every query / key row: padded
 * [B][n_q] and [B][n_k] (row i of batch element b at b * n + i), packed
 * [T_q] and [T_k]; |pos| < 2^24 (see attn_rope).  base finite and > 1
 * (ATTN_ERR_SCALE); NULL positions give ATTN_ERR_NULL.
 * q_rot, k_rot (optional, 16-byte aligned, device): the rotated rows, bf16
 * in Q's and K's contiguous layouts ([B][Hq][n_q][d_h] and
 * [B][Hkv][n_k][d_h]; packed [T_q][Hq][d_h] and [T_k][Hkv][d_h]).  The
 * forward writes its rotated queries and keys there (else into its
 * workspace); a backward given them reads them instead of rotating Q and K
 * again (they must hold what the forward wrote for the same Q, K and
 * positions; the backward's Q and K arguments are then not read for the
 * rows' values).  Keeping them is the trade an unfused rotation makes, which
 * keeps the rotated rows for the attention's backward.  Without them the
 * backward turns Q as it reads it and writes a rotated copy of K into its
 * workspace.  Pass the same rotary to the workspace-size functions: a
 * workspace holds the rotated rows that have no caller buffer.  The decode
 * forward takes no rotary (rotate its few queries with attn_rope; a key
 * cache holds rotated keys). */
typedef struct {
  float base;             /* w_k = base^(-2k/d_h), k < d_h/2                     */
  const int32_t* pos_q;   /* DEVICE positions of the query rows                   */
  const int32_t* pos_k;   /* DEVICE positions of the key rows                     */
  void* q_rot;            /* DEVICE rotated queries, or NULL                      */
  void* k_rot;            /* DEVICE rotated keys, or NULL                         */
} attn_rotary;

/* Bytes of device workspace attn_fwd needs: an fp16 copy of V in 128-key
 * tiles with one exponent per tile, about B*Hkv*ceil(n_k/128)*128*(2*d_v)
 * bytes, plus with a rotary the rotated rows it has no buffer for
 * (B*Hq*n_q*2*d_h bytes of queries, B*Hkv*n_k*2*d_h of keys).  The layout
 * is private to the library.  Returns 0 for an invalid shape or rotary. */
size_t attn_fwd_workspace_bytes(const attn_shape* shape, const attn_rotary* rotary);

/* Forward pass (A.10.1-A.10.3).  Inputs Q, K, V (bf16, device); outputs
 * O (bf16) and LSE (fp32, natural log), both device, fully overwritten.
 * `workspace`: caller-owned device memory of at least
 * attn_fwd_workspace_bytes(shape) bytes, 256-byte aligned (ATTN_ERR_WORKSPACE
 * otherwise); its contents on entry do not matter.  Two launches on
 * `stream`: V re-encoded into the workspace (with a rotary, the same launch
 * writes the rotated queries and keys), then the forward kernel.
 *
 * O_lo (optional here, NULL to skip; required by the backward): bf16
 * [B][Hq][n_q][d_v] receiving the rounding residual of O, so that O + O_lo
 * carries the fp32 result to about 16 significant bits.  The backward's row
 * term c_i = sum_l dO_il O_il (A.10.7) feeds dQ_i with weight
 * -scale * sum_j A_ij k_j, which for a sharply peaked softmax row is a whole
 * key row; bf16 rounding of O alone then moves dQ and dK beyond the stated
 * tolerance (measured: up to 2.2x on the peaked cross-attention workload,
 * 4x on smaller peaked cases). */
int attn_fwd(const attn_shape* shape, const attn_mask* mask, const attn_strides* strides,
             const attn_rotary* rotary, float scale,
             const void* Q, const void* K, const void* V,
             void* O, float* LSE, void* O_lo,
             void* workspace, size_t workspace_bytes, void* stream);

/* Forward for short query blocks over a long key cache (decode, small
 * chunks of new queries: the new-queries-over-a-history shape of "Chapter
 * 31", section 1), n_q <= 128.  Same function, arguments and outputs as
 * attn_fwd (A.10.1-A.10.3, same visible sets); the work is laid out
 * differently: the query heads that share a KV head are packed into one
 * 128-row tile, so each K/V tile is read once per group, and the key range is
 * split across CTAs, the partial results being merged by their log-sum-exp
 * (O = sum_s exp(LSE_s - LSE) O_s, LSE = log sum_s exp(LSE_s)).
 * `workspace`: device memory of at least attn_fwd_decode_workspace_bytes()
 * bytes, 256-byte aligned (may be NULL when that is 0).  Returns
 * ATTN_ERR_UNSUPPORTED for n_q > 128 (use attn_fwd).  Tensors contiguous. */
size_t attn_fwd_decode_workspace_bytes(const attn_shape* shape, const attn_mask* mask);
int attn_fwd_decode(const attn_shape* shape, const attn_mask* mask, float scale,
                    const void* Q, const void* K, const void* V,
                    void* O, float* LSE, void* O_lo,
                    void* workspace, size_t workspace_bytes, void* stream);

/* Bytes of device workspace the backward needs (attn_bwd and its three
 * stages): row terms D, per-128-row-tile bounds used to scale dS, the main
 * kernel's work counter, an fp32 dQ accumulator and fp16 copies of Q and
 * dO, about B*Hq*n_q*(6*d_h + 2*d_v + 4) bytes, plus with a rotary and no k_rot a
 * rotated copy of K, B*Hkv*n_k*2*d_h bytes, plus, when the KV head groups
 * have several query heads and B*Hkv*ceil(n_k/128) < 304 (a launch that
 * may split them, see attn_bwd_head_split), fp32 sums of dK and dV,
 * B*Hkv*n_k*4*(d_h + d_v) bytes.
 * The layout is private to the library.  Returns 0 for an invalid shape or
 * rotary. */
size_t attn_bwd_workspace_bytes(const attn_shape* shape, const attn_rotary* rotary);

/* Backward pass (A.10.5-A.10.9).  Q, K, V, O, O_lo, LSE must be those of
 * the forward call with the same mask and scale ("Chapter 31", section 3:
 * the backward must use the forward's semantics).  O_lo, the forward's
 * rounding residual of O, is required (ATTN_ERR_NULL when NULL): the row
 * terms c_i are formed from O + O_lo (see attn_fwd).  dO is the upstream
 * gradient.
 * Outputs dQ, dK, dV (bf16, device) are fully overwritten; dK and dV hold the
 * sums over each KV head's query heads.  `workspace` is caller-owned device
 * memory of at least attn_bwd_workspace_bytes(shape) bytes, 256-byte aligned;
 * its contents on entry do not matter.  Equivalent to the three stage calls
 * below, in order, on the same workspace.
 *
 * Precision: every product runs in fp16 with fp32 accumulation: Q, K, V
 * and dO are re-encoded as fp16 tile by tile with their own powers of two
 * (exact at any scale, see Precision above), the weights A are rounded once
 * to fp16, and dS enters dK and dQ in fp16 scaled by a power of two derived
 * from a bound on |dS|. */
int attn_bwd(const attn_shape* shape, const attn_mask* mask, const attn_strides* strides,
             const attn_rotary* rotary, float scale,
             const void* Q, const void* K, const void* V,
             const void* O, const void* O_lo, const void* dO, const float* LSE,
             void* dQ, void* dK, void* dV,
             void* workspace, size_t workspace_bytes, void* stream);

/* Stage 1 of the backward: D_i = sum_l dO_il (O_il + O_lo_il) (= c_i of
 * A.10.7; O_lo required), per-tile bounds max ||dO_i|| and max |D_i|, a
 * zeroed dQ accumulator, a zeroed work counter for stage 2 and Q and dO
 * re-encoded as fp16 with per-tile exponents (see attn_bwd), all in
 * `workspace`.  Q is the forward's bf16 query tensor, dO the bf16 upstream
 * gradient. */
int attn_bwd_preprocess(const attn_shape* shape, const attn_strides* strides, const attn_rotary* rotary,
                        const void* Q, const void* O,
                        const void* O_lo, const void* dO, void* workspace,
                        size_t workspace_bytes, void* stream);

/* Stage 2: the key-tile-stationary main kernel.  Recomputes A from the
 * workspace's fp16 copy of Q (written by stage 1), K and LSE, takes dO from
 * the workspace's fp16 copy (also written by stage 1), writes dK (scaled)
 * and dV (bf16) and adds the dS K products into the workspace's fp32 dQ
 * accumulator (zeroed by stage 1).  Under the persistent schedule (see
 * attn_bwd_persistent) the CTAs take their work items from a counter in
 * the workspace that stage 1 zeroes, so every stage 2 call needs a stage 1
 * call on the same workspace before it (as the dQ accumulator already
 * does). */
int attn_bwd_main(const attn_shape* shape, const attn_mask* mask, const attn_strides* strides,
                  const attn_rotary* rotary, float scale,
                  const void* K, const void* V, const float* LSE,
                  void* workspace, size_t workspace_bytes,
                  void* dK, void* dV, void* stream);

/* Stage 3: dQ = scale * accumulator, rounded to bf16.
 *
 * With a rotary, the three stages take the same one: stage 1 rotates Q as
 * it reads it (or reads q_rot), stage 2 writes the rotated keys into the
 * workspace (one extra launch; or reads k_rot) and turns dK back, stage 3
 * turns dQ back. */
int attn_bwd_finalize(const attn_shape* shape, const attn_strides* strides, const attn_rotary* rotary,
                      float scale, const void* workspace,
                      size_t workspace_bytes, void* dQ, void* stream);

/* The backward pass without any device allocation, for callers that cannot
 * call cudaMalloc where they run it: applications whose device memory is all
 * owned by a fixed arena or by another runtime that forbids further
 * allocations, and latency-critical loops that cannot afford cudaMalloc's
 * implicit device-wide synchronisation.  There is no counterpart on the
 * pages: it is attn_bwd with its workspace taken from a static buffer
 * compiled into the library (attn_bwd_noalloc_max_scratch_bytes() bytes,
 * 16 MiB, held on every GPU that loads the library until the process exits).
 *
 * Arguments and results are those of attn_bwd minus the workspace; the
 * caller still provides every input and output.  A problem whose workspace
 * (attn_bwd_workspace_bytes) exceeds the buffer returns ATTN_ERR_WORKSPACE
 * before anything is launched.  The first call on a device looks up the
 * buffer's device address (cudaGetSymbolAddress, with that device current);
 * make that first call before any stream capture.  Every call shares the one
 * buffer, whose contents persist between calls: the kernels clear what must
 * start at zero, but calls that overlap on the GPU race and must be
 * serialised by the caller. */
int attn_bwd_noalloc(const attn_shape* shape, const attn_mask* mask, const attn_strides* strides,
                     const attn_rotary* rotary, float scale,
                     const void* Q, const void* K, const void* V,
                     const void* O, const void* O_lo, const void* dO, const float* LSE,
                     void* dQ, void* dK, void* dV, void* stream);

/* Size in bytes of the static buffer attn_bwd_noalloc uses. */
size_t attn_bwd_noalloc_max_scratch_bytes(void);

/* How attn_bwd_main divides the work of each KV head on the current
 * device: 1 = one work item per (batch, KV head, key tile), taking every
 * query head of the group ("Appendix A.10", section A.10.5: dK, dV summed
 * over the group); z > 1 = the group's query heads split over z work items,
 * each adding its fp32 share of dK, dV into sums in the workspace that a
 * last launch rounds into dK, dV.  Chosen when there are too few items to
 * keep every SM busy to the end (a long-history MQA chunk: one KV head,
 * few key tiles) and the split is predicted to finish at least 3 % sooner;
 * never with a rotary.  With
 * a split, dK and dV are fp32 sums added in whatever order the CTAs finish
 * (as dQ always is), so two runs may differ in the last bf16 unit.
 * Negative ATTN_ERR_* on an invalid shape or mask.  Informational: the
 * calls choose by themselves. */
int attn_bwd_head_split(const attn_shape* shape, const attn_mask* mask);

/* Which schedule attn_bwd_main runs on the current device (with this
 * rotary, or NULL): 0 = one CTA per work item (batch, KV head, 128-key
 * tile, query-head share), 1 = persistent, one CTA per SM taking the items
 * from a counter in the workspace.  Same arithmetic and results either way
 * (dK, dV bit for bit; dQ's fp32 sums in whatever order the items finish).
 * The persistent schedule hides each item's fixed cost (loads, re-encoding,
 * epilogue: about 3.5 steps' worth) behind its neighbours' steps but runs
 * its steps a little slower, so it is taken when the mean item has at most
 * 40 steps (128-query tiles times query heads).  Negative ATTN_ERR_* on an
 * invalid shape or mask.  Informational. */
int attn_bwd_persistent(const attn_shape* shape, const attn_mask* mask, const attn_rotary* rotary);

/* Number of visible (i, j) pairs over all batch elements and query heads,
 * from the same closed form the kernels use to classify tiles; -1 on an
 * invalid shape or mask.  Host only. */
int64_t attn_visible_pairs(const attn_shape* shape, const attn_mask* mask);

/* Packed variable-length sequences: padding removed on both axes ("Appendix
 * A.10", section A.10.6 removes padding positions from the keys; here the
 * queries of each sequence are only its own).  Sequence b has
 * len_q(b) = cu_seqlens_q[b+1] - cu_seqlens_q[b] queries and
 * len_k(b) = cu_seqlens_k[b+1] - cu_seqlens_k[b] keys, stored token-major:
 *   Q, dQ       [T_q][Hq ][d_h]  bf16     K, dK [T_k][Hkv][d_h] bf16
 *   O, O_lo, dO [T_q][Hq ][d_v]  bf16     V, dV [T_k][Hkv][d_v] bf16
 *   LSE         [Hq][T_q]        fp32
 * with T_q = cu_seqlens_q[B], T_k = cu_seqlens_k[B]; query token cu_q[b] + i
 * is row i of sequence b (the same for keys).  A single sequence with
 * equal lengths is the [S][H][d] layout.  Visible set of row i of sequence
 * b: V_i = { j < len_k(b) }, and when causal j <= i + len_k(b) - len_q(b)
 * (each sequence's last query aligned with its last key).  A sequence with
 * len_q(b) > 0 needs len_k(b) >= 1, and when causal len_k(b) >= len_q(b)
 * (else its first rows are empty: ATTN_ERR_EMPTY_ROW); len_q(b) = 0 is
 * allowed (that sequence's keys then get dK = dV = 0).  Same functions,
 * precision, workspace rules and errors as attn_fwd / attn_bwd. */
typedef struct {
  int32_t B;                    /* sequences, 1..ATTN_MAX_BATCH                     */
  int32_t Hq;                   /* query heads                                      */
  int32_t Hkv;                  /* key/value heads; Hq % Hkv == 0                   */
  int32_t d_h;                  /* query/key width                                  */
  int32_t d_v;                  /* value width                                      */
  int32_t causal;               /* 0 or 1 (bottom-right aligned per sequence)       */
  const int32_t* cu_seqlens_q;  /* HOST [B+1]: 0 = cu[0] <= cu[1] <= ... <= cu[B]    */
  const int32_t* cu_seqlens_k;  /* HOST [B+1], same rules                           */
} attn_varlen;

/* Visible (query, key) pairs over all sequences and query heads, -1 when
 * the description is invalid. */
int64_t attn_varlen_visible_pairs(const attn_varlen* v);

/* Workspace of attn_fwd_varlen, about B*Hkv*ceil(max len_k/128)*128*(2*d_v)
 * bytes (the fp16 V tiles are laid out per sequence), plus with a rotary
 * the rotated rows without a caller buffer ((T_q*Hq + T_k*Hkv)*2*d_h bytes
 * at most); 0 when the description is invalid. */
size_t attn_fwd_varlen_workspace_bytes(const attn_varlen* v, const attn_rotary* rotary);

int attn_fwd_varlen(const attn_varlen* v, const attn_strides* strides, const attn_rotary* rotary, float scale,
                    const void* Q, const void* K,
                    const void* V,
                    void* O, float* LSE, void* O_lo, void* workspace, size_t workspace_bytes, void* stream);

/* Workspace of attn_bwd_varlen, about T_q*Hq*(6*d_h + 2*d_v + 4) bytes; 0 when the
 * description is invalid. */
size_t attn_bwd_varlen_workspace_bytes(const attn_varlen* v, const attn_rotary* rotary);

int attn_bwd_varlen(const attn_varlen* v, const attn_strides* strides, const attn_rotary* rotary, float scale,
                    const void* Q, const void* K,
                    const void* V,
                    const void* O, const void* O_lo, const void* dO, const float* LSE,
                    void* dQ, void* dK, void* dV, void* workspace, size_t workspace_bytes,
                    void* stream);

/* Linear projections on either side of attention ("Appendix A.10", eqs.
 * A.10.10-A.10.11), on the tensor cores.  Row-major matrices, bf16 in, fp32
 * accumulation; T rows (tokens), D input width, N output width (for example
 * Hq * d_h: the output [T][Hq*d_h] is the packed [T][Hq][d_h] layout the
 * variable-length entry points take).
 *   attn_proj_fwd:        Y [T][N] = X [T][D] W [D][N]                 bf16 out
 *   attn_proj_bwd_weight: dW [D][N] = X^T G,  G [T][N]                 fp32 out
 *   attn_proj_bwd_input:  dX [T][D] = sum_s G_s [T][N_s] W_s[D][N_s]^T bf16 out,
 *                         over 1..3 sources: the branches that share X (all
 *                         three for self-attention; only the shared ones for
 *                         cross-attention, A.10.11).  N, G, W are host arrays
 *                         of nsrc entries (G[s], W[s] device pointers).
 * D and every N must be multiples of 8 (16-byte rows): ATTN_ERR_SHAPE
 * otherwise; pointers 16-byte aligned.  Outputs are fully overwritten. */
int attn_proj_fwd(int64_t T, int32_t D, int32_t N, const void* X, const void* W, void* Y, void* stream);
int attn_proj_bwd_weight(int64_t T, int32_t D, int32_t N, const void* X, const void* G, float* dW,
                         void* stream);
int attn_proj_bwd_input(int64_t T, int32_t D, int32_t nsrc, const int32_t* N, const void* const* G,
                        const void* const* W, void* dX, void* stream);

/* Rotary position embedding of query or key rows ("Chapter 15 -- matrix
 * formulas", section 15.6): every row x of width d is split into 2-D blocks
 * (x_2k, x_2k+1), k < d/2, and block k is rotated by a = pos * w_k with
 * w_k = base^(-2k/d) (column-vector rotation: x'_2k = x_2k cos a - x_2k+1
 * sin a, x'_2k+1 = x_2k sin a + x_2k+1 cos a), so that the score of a rotated
 * query and key depends only on their position difference.  inverse = 1
 * rotates by -a: the transpose, which maps the gradient of a rotated row back
 * to the row ("Chapter 31 -- attention backprop", section 5).
 * X, Y: device bf16 [tokens][heads][d] (token-major, the packed layout; Y may
 * equal X); positions: device int32 [tokens], the position of each token.
 * d a multiple of 8 and <= 128; base finite and > 1 (ATTN_ERR_SCALE
 * otherwise).  Positions must satisfy |pos| < 2^24 (the integers an fp32
 * holds exactly).  Each frequency reaches the kernel as an fp32 value plus
 * its rounding residual, the product pos * w keeps its own rounding
 * residual, and the angle is reduced modulo 2 pi in three steps, so the
 * angle is accurate to a few 1e-7 rad over that whole range (tested against
 * exact fp64 angles for positions up to 2^24 - 1). */
int attn_rope(int64_t tokens, int32_t heads, int32_t d, float base, const int32_t* positions, int32_t inverse,
              const void* X, void* Y, void* stream);

/* The rotation of a batch's queries and keys in one launch: Xq, Yq are
 * [tokens][heads_q][d], Xk, Yk [tokens][heads_k][d], both at the same
 * positions.  Equal, bit for bit, to attn_rope on Xq followed by attn_rope
 * on Xk with the same tokens, d, base, positions and inverse; the argument
 * rules and errors are those of attn_rope, for both tensors (Yq may equal Xq
 * and Yk may equal Xk; no other overlap is allowed).  One launch instead of
 * two: the keys' short pass does not pay a launch, a ramp and a tail of its
 * own. */
int attn_rope_qk(int64_t tokens, int32_t heads_q, int32_t heads_k, int32_t d, float base,
                 const int32_t* positions, int32_t inverse, const void* Xq, void* Yq, const void* Xk, void* Yk,
                 void* stream);

/* Device status word of the current device: ATTN_OK, or the first failure a
 * kernel recorded (ATTN_ERR_TIMEOUT).  Synchronises the device.  Writes the
 * status to *status and returns ATTN_OK, or ATTN_ERR_CUDA. */
int attn_get_status(int* status);

/* Reset the device status word to ATTN_OK.  Synchronises the device. */
int attn_clear_status(void);

/* Failure-detection self test: launches one tiny kernel that waits on a
 * barrier nothing will complete, with a limit of `limit_ns` nanoseconds, so
 * the bounded-wait path records ATTN_ERR_TIMEOUT in the status word and the
 * kernel returns.  Enqueued on `stream`. */
int attn_selftest_wait_timeout(uint64_t limit_ns, void* stream);

/* Human-readable name of a status code (static string). */
const char* attn_strerror(int status);

/* ATTN_ABI_VERSION of the loaded library. */
int attn_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* EXACT_SCALED_DOT_GB300_ATTN_H */
