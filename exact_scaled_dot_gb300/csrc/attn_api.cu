// attn_api.cu -- the C ABI (include/attn.h): argument validation, TMA tensor
// descriptors, launches, the device status word and the failure-detection
// self test.  Every argument check runs before the first CUDA call, so an
// invalid call returns its error code without touching the GPU.
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <functional>
#include <mutex>
#include <queue>
#include <vector>

#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/attn.h"
#include "common.cuh"
#include "f16range.cuh"
#include "ptx.cuh"

namespace esd {
namespace {

// Device status word: ATTN_OK, or the first failure a kernel recorded.
__device__ unsigned int g_attn_status = 0u;

constexpr int kMaxDevices = 64;

// ---------------------------------------------------------------------------
// Validation (host only, no CUDA calls)
// ---------------------------------------------------------------------------
bool supported_dims(int dh, int dv) {
  return (dh == 64 && dv == 64) || (dh == 128 && dv == 128) || (dh == 128 && dv == 64);
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_shape(const attn_shape* s) {
  if (!s) return ATTN_ERR_NULL;
  if (s->B <= 0 || s->Hq <= 0 || s->Hkv <= 0 || s->n_q <= 0 || s->n_k <= 0 || s->d_h <= 0 || s->d_v <= 0)
    return ATTN_ERR_SHAPE;
  if (s->Hq % s->Hkv != 0) return ATTN_ERR_SHAPE;
  if (s->B > ATTN_MAX_BATCH) return ATTN_ERR_SHAPE;
  // Grid and index limits: (B*Hq) blocks along x; element counts fit int64.
  const int64_t bhq = static_cast<int64_t>(s->B) * s->Hq;
  if (bhq > (int64_t{1} << 31) - 1) return ATTN_ERR_SHAPE;
  // Grid dimensions y: forward query-tile pairs, preprocess query tiles and
  // backward key tiles must stay within 65535.
  if ((static_cast<int64_t>(s->n_k) + 127) / 128 > 65535) return ATTN_ERR_SHAPE;
  if ((static_cast<int64_t>(s->n_q) + 127) / 128 > 65535) return ATTN_ERR_SHAPE;
  if (!supported_dims(s->d_h, s->d_v)) return ATTN_ERR_UNSUPPORTED;
  return ATTN_OK;
}

// Effective mask parameters.  The visible set of row i in batch b is
// { j < kv_len[b] } intersected, when causal, with { j <= i + offset }.
// Because both bounds only grow with i, every row is non-empty iff row 0 is:
// kv_len[b] >= 1 for every b and, when causal, offset >= 0.
int build_mask(const attn_shape* s, const attn_mask* m, MaskParams* out) {
  std::memset(out, 0, sizeof(*out));
  if (!m) return ATTN_ERR_NULL;
  if (m->reserved != 0 || (m->causal != 0 && m->causal != 1)) return ATTN_ERR_SHAPE;
  out->causal = m->causal;
  if (m->kv_len) {
    out->has_kv_len = 1;
    for (int b = 0; b < s->B; ++b) {
      const int32_t L = m->kv_len[b];
      if (L < 0 || L > s->n_k) return ATTN_ERR_SHAPE;
      if (L == 0) return ATTN_ERR_EMPTY_ROW;
      out->kv_len[b] = L;
    }
  }
  if (m->causal) {
    int64_t off = (m->causal_offset == ATTN_OFFSET_DEFAULT)
                      ? static_cast<int64_t>(s->n_k) - static_cast<int64_t>(s->n_q)
                      : m->causal_offset;
    if (off < 0) return ATTN_ERR_EMPTY_ROW;
    if (off > s->n_k) off = s->n_k;   // beyond n_k the causal bound never binds
    out->offset = off;
  }
  return ATTN_OK;
}

int check_scale(float scale) {
  return (std::isfinite(scale) && scale > 0.f) ? ATTN_OK : ATTN_ERR_SCALE;
}

int check_ptrs(std::initializer_list<const void*> ptrs) {
  for (const void* p : ptrs)
    if (!p) return ATTN_ERR_NULL;
  for (const void* p : ptrs)
    if (!aligned16(p)) return ATTN_ERR_ALIGN;
  return ATTN_OK;
}

size_t round256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// One tensor's strides: the caller's ({0, 0} = contiguous), checked.
int one_strides(const attn_tensor_strides* user, int64_t row0, int64_t head0, int d, TensorStrides* out) {
  if (!user || (user->row == 0 && user->head == 0)) {
    *out = TensorStrides{row0, head0};
    return ATTN_OK;
  }
  if (user->row % 8 != 0 || user->head % 8 != 0) return ATTN_ERR_ALIGN;
  if (user->row < d || user->head < d || user->row > (int64_t{1} << 36) || user->head > (int64_t{1} << 36))
    return ATTN_ERR_SHAPE;
  *out = TensorStrides{user->row, user->head};
  return ATTN_OK;
}

// Every user tensor's strides into `lay` (whose `packed` is set): padded
// [B][H][n][d] defaults row = d, head = n d; packed [T][H][d] defaults
// row = H d, head = d.
int build_strides(const attn_strides* st, int Hq, int Hkv, int n_q, int n_k, int dh, int dv, LayoutParams* lay) {
  const bool pk = lay->packed != 0;
  auto def = [&](int H, int n, int d, int64_t& row, int64_t& head) {
    row = pk ? static_cast<int64_t>(H) * d : d;
    head = pk ? d : static_cast<int64_t>(n) * d;
  };
  struct Item {
    const attn_tensor_strides* user;
    TensorStrides* out;
    int H, n, d;
  } items[8] = {{st ? &st->q : nullptr, &lay->sq, Hq, n_q, dh},   {st ? &st->k : nullptr, &lay->sk, Hkv, n_k, dh},
                {st ? &st->v : nullptr, &lay->sv, Hkv, n_k, dv},  {st ? &st->o : nullptr, &lay->so, Hq, n_q, dv},
                {st ? &st->dO : nullptr, &lay->sdo, Hq, n_q, dv}, {st ? &st->dq : nullptr, &lay->sdq, Hq, n_q, dh},
                {st ? &st->dk : nullptr, &lay->sdk, Hkv, n_k, dh}, {st ? &st->dv : nullptr, &lay->sdv, Hkv, n_k, dv}};
  for (const Item& it : items) {
    int64_t row, head;
    def(it.H, it.n, it.d, row, head);
    const int rc = one_strides(it.user, row, head, it.d, it.out);
    if (rc) return rc;
  }
  return ATTN_OK;
}

// Whether a tensor has its layout's contiguous strides.
bool contiguous_strides(const LayoutParams& lay, const TensorStrides& s, int H, int n, int d) {
  return lay.packed ? (s.row == static_cast<int64_t>(H) * d && s.head == d)
                    : (s.row == d && s.head == static_cast<int64_t>(n) * d);
}

// Sum over query rows of max(0, lim(b, i)) for one batch element.
int64_t pairs_one_batch(const MaskParams& m, int n_q, int n_k, int b) {
  const int64_t L = key_len(m, n_k, b);
  const int64_t nq = query_len(m, n_q, b);
  if (!m.causal) return L * nq;
  // Rows with i + offset + 1 < L see i + offset + 1 keys; the rest see L.
  const int64_t off = causal_offset(m, b);
  int64_t split = L - off - 1;             // rows i < split are causal-bound
  if (split < 0) split = 0;
  if (split > nq) split = nq;
  const int64_t head = split * (off + 1) + split * (split - 1) / 2;
  return head + (nq - split) * L;
}

// A packed variable-length description turned into the kernels' terms: the
// shape's n_q, n_k are the longest sequence (grid extents), the mask carries
// every sequence's lengths and its own bottom-right causal offset, and the
// layout its token offsets.
struct Varlen {
  attn_shape shape;
  MaskParams mask;
  LayoutParams lay;
  int64_t total_q, total_k;
};

int build_varlen(const attn_varlen* v, Varlen* out) {
  if (!v || !v->cu_seqlens_q || !v->cu_seqlens_k) return ATTN_ERR_NULL;
  if (v->B <= 0 || v->B > ATTN_MAX_BATCH || v->Hq <= 0 || v->Hkv <= 0 || v->d_h <= 0 || v->d_v <= 0)
    return ATTN_ERR_SHAPE;
  if (v->Hq % v->Hkv != 0 || (v->causal != 0 && v->causal != 1)) return ATTN_ERR_SHAPE;
  if (!supported_dims(v->d_h, v->d_v)) return ATTN_ERR_UNSUPPORTED;
  if (v->cu_seqlens_q[0] != 0 || v->cu_seqlens_k[0] != 0) return ATTN_ERR_SHAPE;
  std::memset(out, 0, sizeof(*out));
  int32_t max_q = 0, max_k = 0;
  for (int b = 0; b < v->B; ++b) {
    const int64_t lq = static_cast<int64_t>(v->cu_seqlens_q[b + 1]) - v->cu_seqlens_q[b];
    const int64_t lk = static_cast<int64_t>(v->cu_seqlens_k[b + 1]) - v->cu_seqlens_k[b];
    if (lq < 0 || lk < 0) return ATTN_ERR_SHAPE;
    if (lq > 0 && lk == 0) return ATTN_ERR_EMPTY_ROW;
    if (v->causal && lq > lk) return ATTN_ERR_EMPTY_ROW;   // row 0 would see keys j <= lk - lq < 0
    out->mask.kv_len[b] = static_cast<int32_t>(lk);
    out->mask.q_len[b] = static_cast<int32_t>(lq);
    max_q = std::max<int32_t>(max_q, static_cast<int32_t>(lq));
    max_k = std::max<int32_t>(max_k, static_cast<int32_t>(lk));
  }
  out->mask.causal = v->causal;
  out->mask.has_kv_len = 1;
  out->mask.has_q_len = 1;
  out->mask.offset_from_lengths = 1;
  out->lay.packed = 1;
  for (int b = 0; b <= v->B; ++b) {
    out->lay.cu_q[b] = v->cu_seqlens_q[b];
    out->lay.cu_k[b] = v->cu_seqlens_k[b];
  }
  out->total_q = v->cu_seqlens_q[v->B];
  out->total_k = v->cu_seqlens_k[v->B];
  out->lay.total_q = out->total_q;
  // Grid extents from the longest sequence (at least one tile).
  out->shape = attn_shape{v->B, v->Hq, v->Hkv, std::max(max_q, 1), std::max(max_k, 1), v->d_h, v->d_v};
  if ((static_cast<int64_t>(out->shape.n_k) + 127) / 128 > 65535) return ATTN_ERR_SHAPE;
  if ((static_cast<int64_t>(out->shape.n_q) + 127) / 128 > 65535) return ATTN_ERR_SHAPE;
  return ATTN_OK;
}

// ---------------------------------------------------------------------------
// CUDA-side helpers
// ---------------------------------------------------------------------------
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*,
                                   CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                   CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
  });
  return fn;
}

// 3-D view [bh][n][d] of a tensor of 2-byte elements (bf16, or the
// backward's fp16 copy of Q: the copy does not interpret the values) with
// element strides row (default d) and head (default n d), read in 128-row x
// 64-col boxes with the 128-byte swizzle the tensor-core operand layout
// expects.  Rows beyond n of a head read as all-zero bits (bounds fill, 0 in
// either type), never the next head.
bool make_tmap(CUtensorMap* map, const void* ptr, int d, int n, int64_t bh, int64_t row_stride = 0,
               int64_t head_stride = 0) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  if (row_stride == 0) row_stride = d;
  if (head_stride == 0) head_stride = static_cast<int64_t>(n) * d;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(n), static_cast<cuuint64_t>(bh)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(row_stride) * 2, static_cast<cuuint64_t>(head_stride) * 2};
  cuuint32_t box[3] = {64, 128, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D view [bh][n][d] of the fp32 dQ accumulator for TMA reduce-add in
// 32-row x 32-column boxes (128-byte rows, 128-byte swizzle); rows beyond n
// of a head are clipped.
// Token-major view [T][H][d] (packed sequences) of a 2-byte tensor with
// element strides row (between tokens, default H d) and head (default d):
// dims (d, H, T), boxes of 64 columns x 1 head x 128 tokens, which land in
// shared memory exactly like the padded view's 128-row x 64-col boxes.
// Tokens past T read as zeros.
bool make_tmap_packed(CUtensorMap* map, const void* ptr, int d, int H, int64_t T, int64_t row_stride = 0,
                      int64_t head_stride = 0) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  if (row_stride == 0) row_stride = static_cast<int64_t>(H) * d;
  if (head_stride == 0) head_stride = d;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(T)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(head_stride) * 2, static_cast<cuuint64_t>(row_stride) * 2};
  cuuint32_t box[3] = {64, 1, 128};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The same token-major view of the fp32 dQ accumulator, in boxes of 32
// columns x 1 head x 32 tokens for TMA reduce-add.
bool make_tmap_acc_packed(CUtensorMap* map, const void* ptr, int d, int H, int64_t T) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(T)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 4, static_cast<cuuint64_t>(H) * d * 4};
  cuuint32_t box[3] = {32, 1, 32};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(ptr), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_tmap_acc(CUtensorMap* map, const void* ptr, int d, int n, int64_t bh) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(n), static_cast<cuuint64_t>(bh)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 4, static_cast<cuuint64_t>(n) * d * 4};
  cuuint32_t box[3] = {32, 32, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(ptr), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D view of a row-major [rows][cols] bf16 matrix, boxes of box_cols x
// box_rows with the 128-byte swizzle; rows and columns past the edges read as
// zeros.
bool make_tmap_2d(CUtensorMap* map, const void* ptr, int64_t rows, int64_t cols, int box_cols, int box_rows) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 2};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int check_proj_dims(int64_t T, int32_t D, int32_t N) {
  if (T <= 0 || D <= 0 || N <= 0) return ATTN_ERR_SHAPE;
  if (D % 8 != 0 || N % 8 != 0) return ATTN_ERR_SHAPE;                 // 16-byte rows
  if (T > (int64_t{1} << 31) - 1) return ATTN_ERR_SHAPE;               // TMA coordinates are int32
  if ((T + 127) / 128 > 65535 || (static_cast<int64_t>(D) + 127) / 128 > 65535) return ATTN_ERR_SHAPE;
  return ATTN_OK;
}

struct DeviceInfo {
  bool probed = false;
  bool ok = false;
  unsigned int* status = nullptr;
  int sms = 0;
};

std::mutex g_dev_mu;
DeviceInfo g_dev[kMaxDevices];

// Checks that the current device is an sm_103 GPU and returns the device
// address of its status word.
int device_status_ptr(unsigned int** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return ATTN_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return ATTN_ERR_DEVICE;
  std::lock_guard<std::mutex> lock(g_dev_mu);
  DeviceInfo& d = g_dev[dev];
  if (!d.probed) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return ATTN_ERR_CUDA;
    void* sym = nullptr;
    if (major == 10 && minor == 3) {
      if (cudaGetSymbolAddress(&sym, g_attn_status) != cudaSuccess) return ATTN_ERR_CUDA;
      if (cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return ATTN_ERR_CUDA;
      d.status = static_cast<unsigned int*>(sym);
      d.ok = true;
    }
    d.probed = true;
  }
  if (!d.ok) return ATTN_ERR_DEVICE;
  *out = d.status;
  return ATTN_OK;
}

// SMs of the current device (after device_status_ptr succeeded on it).
int device_sms() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 148;
  std::lock_guard<std::mutex> lock(g_dev_mu);
  return g_dev[dev].sms > 0 ? g_dev[dev].sms : 148;
}

ShapeParams shape_params(const attn_shape* s) {
  ShapeParams sp;
  sp.B = s->B;
  sp.Hq = s->Hq;
  sp.Hkv = s->Hkv;
  sp.n_q = s->n_q;
  sp.n_k = s->n_k;
  sp.group = s->Hq / s->Hkv;
  return sp;
}

int64_t q_rows(const attn_shape* s) { return static_cast<int64_t>(s->B) * s->Hq * s->n_q; }

// Backward workspace: D [rows] | per-query-tile maxima and fp16 exponents
// float4 [B*Hq*nqt] | per-group fp16 exponents float2 [B*Hkv] | the main
// kernel's work counter (256 bytes) | fp32 dQ accumulator [rows * d_h] |
// fp16 copy of Q [rows * d_h] | fp16 copy of dO [rows * d_v], each 256-byte
// aligned.
// With a rotary, then the rotated keys bf16 [tokens_k Hkv][d_h]
// (contiguous in the keys' layout).  When the launch may split a KV head's
// query heads across CTAs (head_split_possible), then the fp32 sums of dK
// and dV, [tokens_k Hkv][d_h] and [tokens_k Hkv][d_v], one after the other.
struct Workspace {
  float* D;
  float4* tilemax;
  float2* grpexp;
  unsigned int* work_ctr;
  float* dQacc;
  void* Q16;
  void* dO16;
  void* Kr;
  float* dKacc;
  float* dVacc;
  size_t kv_elems;
  size_t bytes;
};

// A query-head split is considered when the KV head groups have several
// query heads and the launch has fewer than two CTAs per SM of the largest
// part (152 SMs): longer launches fill the GPU by themselves.
constexpr int64_t kSplitCtaLimit = 2 * 152;

bool head_split_possible(int B, int Hq, int Hkv, int n_k) {
  const int64_t ctas = static_cast<int64_t>(B) * Hkv * ((n_k + kTileN - 1) / kTileN);
  return Hq / Hkv > 1 && ctas < kSplitCtaLimit;
}

// The backward main kernel's plan: its schedule (one CTA per work item, or
// persistent CTAs taking items from a counter) and the query-head split z
// (1, or a divisor of the group up to 16 that splits each KV head's query
// heads over z items).
struct BwdPlan {
  int hsplit;
  bool persistent;
};

// Items whose mean step count (128-query tiles times query heads) exceeds
// this run on the grid kernel: its steps are some 5-10 % faster, and with
// this many steps its fixed cost per item (about 3.5 steps) matters less
// than that.  Measured crossover on GB300: persistent ahead with 4, 8.5
// and 33 steps per item, the grid kernel with 62 and 80.
constexpr double kPersistentMaxSteps = 40.0;

// The split z is the one predicted to finish first, by at least 3 %.  The
// prediction hands the items out in the order the schedule starts them to
// whichever of `sms` CTAs frees first.  Grid: in launch order (blockIdx.x,
// the (batch, KV head) index, fastest, then the key tile, then z), an item
// costing its visible (query tile, head) steps plus 5 steps of set-up and
// epilogue (7 when it adds its dK, dV share into the sums).  Persistent: in
// item number order ((batch, KV head) fastest, then z, then the key tile),
// as the work counter hands them out, plus one step of hand-over between
// items (two with the sums).
BwdPlan choose_bwd_plan(const attn_shape* s, const MaskParams& m, int sms, bool rotary) {
  const int group = s->Hq / s->Hkv;
  const int nkt = (s->n_k + kTileN - 1) / kTileN;
  const int bk_n = s->B * s->Hkv;
  // Visible query tiles of key tile jt of batch element b.
  std::vector<int> vis(static_cast<size_t>(s->B) * nkt);
  double steps = 0.0, active = 0.0;
  for (int b = 0; b < s->B; ++b) {
    const int64_t nq_b = query_len(m, s->n_q, b);
    const int nqt = static_cast<int>((nq_b + kTileM - 1) / kTileM);
    for (int jt = 0; jt < nkt; ++jt) {
      const int64_t i_first = first_row_seeing_key(m, s->n_q, s->n_k, b, static_cast<int64_t>(jt) * kTileN);
      const int v = i_first < nq_b ? nqt - static_cast<int>(i_first / kTileM) : 0;
      vis[static_cast<size_t>(b) * nkt + jt] = v;
      steps += static_cast<double>(v) * group * s->Hkv;
      active += v > 0 ? s->Hkv : 0;
    }
  }
  auto makespan = [&](int z, bool persistent) {
    std::priority_queue<double, std::vector<double>, std::greater<double>> free_at;
    for (int i = 0; i < sms; ++i) free_at.push(0.0);
    double end = 0.0;
    const double fixed = persistent ? (z > 1 ? 2.0 : 1.0) : (z > 1 ? 7.0 : 5.0);
    auto take = [&](int jt, int bk) {
      const int b = bk / s->Hkv;
      const double t = free_at.top() + vis[static_cast<size_t>(b) * nkt + jt] * (group / z) + fixed;
      free_at.pop();
      free_at.push(t);
      end = std::max(end, t);
    };
    if (persistent) {
      for (int jt = 0; jt < nkt; ++jt)
        for (int zz = 0; zz < z; ++zz)
          for (int bk = 0; bk < bk_n; ++bk) take(jt, bk);
    } else {
      for (int zz = 0; zz < z; ++zz)
        for (int jt = 0; jt < nkt; ++jt)
          for (int bk = 0; bk < bk_n; ++bk) take(jt, bk);
    }
    return end;
  };
  const bool may_split = !rotary && head_split_possible(s->B, s->Hq, s->Hkv, s->n_k);
  auto best_split = [&](bool persistent) {
    if (!may_split) return 1;   // (no simulation: large launches pay nothing here)
    int best = 1;
    double best_t = makespan(1, persistent);
    const double base_t = best_t;
    for (int z = 2; z <= std::min(group, 16); ++z) {
      if (group % z) continue;
      const double t = makespan(z, persistent);
      if (t < best_t) {
        best_t = t;
        best = z;
      }
    }
    return best_t < 0.97 * base_t ? best : 1;
  };
  const int z_grid = best_split(false);
  const double mean_steps = active > 0.0 ? steps / (active * z_grid) : 0.0;
  if (mean_steps > kPersistentMaxSteps) return BwdPlan{z_grid, false};
  return BwdPlan{best_split(true), true};
}

// The rotary part of a workspace: tokens of the queries and keys (padded
// B n, packed T), and which rotated rows live in the workspace (those
// without a caller buffer).
struct RotaryTokens {
  bool on;
  int64_t q, k;
  bool q_ws, k_ws;
};

// rows: query rows over all heads (B Hq n_q padded, T_q Hq packed); the
// tile bounds are indexed [B Hq][ceil(n_q / 128)] in both layouts.
Workspace workspace_layout_rows(const attn_shape* s, size_t rows, void* base, const RotaryTokens& rt) {
  const size_t nqt = (static_cast<size_t>(s->n_q) + 127) / 128;
  const size_t tiles = static_cast<size_t>(s->B) * s->Hq * nqt;
  const size_t off_t = round256(rows * sizeof(float));
  const size_t off_g = off_t + round256(tiles * sizeof(float4));
  const size_t off_c = off_g + round256(static_cast<size_t>(s->B) * s->Hkv * sizeof(float2));
  const size_t off_a = off_c + 256;
  const size_t off_q = off_a + round256(rows * static_cast<size_t>(s->d_h) * sizeof(float));
  const size_t off_o = off_q + round256(rows * static_cast<size_t>(s->d_h) * 2);
  Workspace w;
  uint8_t* b = static_cast<uint8_t*>(base);
  w.D = reinterpret_cast<float*>(b);
  w.tilemax = reinterpret_cast<float4*>(b + off_t);
  w.grpexp = reinterpret_cast<float2*>(b + off_g);
  w.work_ctr = reinterpret_cast<unsigned int*>(b + off_c);
  w.dQacc = reinterpret_cast<float*>(b + off_a);
  w.Q16 = b + off_q;
  w.dO16 = b + off_o;
  size_t end = off_o + round256(rows * static_cast<size_t>(s->d_v) * 2);
  w.Kr = nullptr;
  if (rt.on && rt.k_ws) {
    w.Kr = b + end;
    end += round256(static_cast<size_t>(rt.k) * s->Hkv * s->d_h * 2);
  }
  w.dKacc = w.dVacc = nullptr;
  w.kv_elems = 0;
  if (head_split_possible(s->B, s->Hq, s->Hkv, s->n_k)) {
    const size_t kv_rows = static_cast<size_t>(rt.k) * s->Hkv;
    w.dKacc = reinterpret_cast<float*>(b + end);
    w.dVacc = w.dKacc + kv_rows * s->d_h;
    w.kv_elems = kv_rows * (s->d_h + s->d_v);
    end += round256(w.kv_elems * sizeof(float));
  }
  w.bytes = end;
  return w;
}

// The persistent schedule's launch (unused by the grid schedule): one work
// item per (batch, KV head, 128-key tile) and query-head share, one CTA per
// SM (fewer when there are fewer items).  Needs p->sh and p->hsplit.  False when the item numbers
// would not fit the kernel's int arithmetic (more than 2^30 items).
bool set_bwd_schedule(BwdParams* p, const Workspace& w, int sms) {
  const int64_t nkt = (p->sh.n_k + kTileN - 1) / kTileN;
  const int64_t items = static_cast<int64_t>(p->sh.B) * p->sh.Hkv * nkt * p->hsplit;
  if (items > (int64_t{1} << 30)) return false;
  p->work_ctr = w.work_ctr;
  p->nitems = static_cast<int32_t>(items);
  p->ctas = static_cast<int32_t>(std::min<int64_t>(items, sms));
  return true;
}

RotaryTokens rotary_tokens(const attn_rotary* r, int64_t q, int64_t k) {
  return RotaryTokens{r != nullptr, q, k, r != nullptr && r->q_rot == nullptr, r != nullptr && r->k_rot == nullptr};
}

RotaryTokens padded_tokens(const attn_shape* s, const attn_rotary* r) {
  return rotary_tokens(r, static_cast<int64_t>(s->B) * s->n_q, static_cast<int64_t>(s->B) * s->n_k);
}

RotaryTokens varlen_tokens(const Varlen& v, const attn_rotary* r) { return rotary_tokens(r, v.total_q, v.total_k); }

Workspace workspace_layout(const attn_shape* s, void* base, const attn_rotary* r) {
  return workspace_layout_rows(s, static_cast<size_t>(q_rows(s)), base, padded_tokens(s, r));
}

Workspace workspace_layout_varlen(const Varlen& v, void* base, const attn_rotary* r) {
  return workspace_layout_rows(&v.shape, static_cast<size_t>(v.total_q) * v.shape.Hq, base, varlen_tokens(v, r));
}

// Forward workspace: the fp16 V tiles [B Hkv][nkt 128][d_v] | their
// exponents int32 [B Hkv][nkt] | with a rotary, the rotated queries bf16
// [tokens_q Hq][d_h] and keys [tokens_k Hkv][d_h] (contiguous in their
// layouts) that have no caller buffer; each 256-byte aligned.  Qr, Kr point
// at wherever the rotated rows go (a caller buffer or the workspace).
struct FwdWorkspace {
  void* V16;
  int32_t* vexp;
  void* Qr;
  void* Kr;
  int nkt;
  size_t bytes;
};

FwdWorkspace fwd_workspace_layout(const attn_shape* s, void* base, const RotaryTokens& rt) {
  FwdWorkspace w;
  w.nkt = (s->n_k + kTileN - 1) / kTileN;
  const size_t tiles = static_cast<size_t>(s->B) * s->Hkv * w.nkt;
  const size_t v16 = round256(tiles * kTileN * static_cast<size_t>(s->d_v) * 2);
  uint8_t* b = static_cast<uint8_t*>(base);
  w.V16 = b;
  w.vexp = reinterpret_cast<int32_t*>(b + v16);
  size_t end = v16 + round256(tiles * sizeof(int32_t));
  w.Qr = w.Kr = nullptr;
  if (rt.on && rt.q_ws) {
    w.Qr = b + end;
    end += round256(static_cast<size_t>(rt.q) * s->Hq * s->d_h * 2);
  }
  if (rt.on && rt.k_ws) {
    w.Kr = b + end;
    end += round256(static_cast<size_t>(rt.k) * s->Hkv * s->d_h * 2);
  }
  w.bytes = end;
  return w;
}

int check_fwd_workspace(const attn_shape* s, const RotaryTokens& rt, const void* ws, size_t bytes) {
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return ATTN_ERR_WORKSPACE;
  if (bytes < fwd_workspace_layout(s, nullptr, rt).bytes) return ATTN_ERR_WORKSPACE;
  return ATTN_OK;
}

// A rotary description: base finite and > 1, both position arrays present
// and 4-byte aligned.  NULL (no rotary) passes.
int check_rotary(const attn_rotary* r) {
  if (!r) return ATTN_OK;
  if (!std::isfinite(r->base) || !(r->base > 1.f)) return ATTN_ERR_SCALE;
  if (!r->pos_q || !r->pos_k) return ATTN_ERR_NULL;
  if ((reinterpret_cast<uintptr_t>(r->pos_q) & 3u) != 0 || (reinterpret_cast<uintptr_t>(r->pos_k) & 3u) != 0)
    return ATTN_ERR_ALIGN;
  if ((r->q_rot && !aligned16(r->q_rot)) || (r->k_rot && !aligned16(r->k_rot))) return ATTN_ERR_ALIGN;
  return ATTN_OK;
}

// Frequencies w_k = base^(-2k/d) in double, passed as fp32 pairs w_hi + w_lo
// so that the rounding of w does not grow with the position.
void rope_frequencies(float base, int d, float* w_hi, float* w_lo) {
  for (int k = 0; k < d / 2; ++k) {
    const double w = std::pow(static_cast<double>(base), -2.0 * k / d);
    w_hi[k] = static_cast<float>(w);
    w_lo[k] = static_cast<float>(w - static_cast<double>(w_hi[k]));
  }
}

// One segment of rotated rows ahead of the attention kernels: `tokens`
// rows of X's H heads at positions pos, written contiguous into Y (an empty
// segment when Y is nullptr).
RopeSegment rope_segment(int64_t tokens, int n, int H, const int32_t* pos, const void* X, const TensorStrides& sx,
                         void* Y) {
  RopeSegment g;
  std::memset(&g, 0, sizeof(g));
  g.tokens = Y ? tokens : 0;
  g.n = n;
  g.H = H;
  g.pos = pos;
  g.X = X;
  g.sx = sx;
  g.Y = Y;
  return g;
}

RopePrepParams rotary_prep(const attn_rotary* r, int d, bool packed, const RopeSegment& a, const RopeSegment& b) {
  RopePrepParams p;
  std::memset(&p, 0, sizeof(p));
  p.d = d;
  p.packed = packed ? 1 : 0;
  p.seg[0] = a;
  p.seg[1] = b;
  rope_frequencies(r->base, d, p.w_hi, p.w_lo);
  return p;
}

// Positions and frequencies for a kernel that turns rows itself.
RotaryAngles rotary_angles(const attn_rotary* r, const int32_t* pos, int d) {
  RotaryAngles a;
  std::memset(&a, 0, sizeof(a));
  a.pos = pos;
  rope_frequencies(r->base, d, a.w_hi, a.w_lo);
  return a;
}

int launch_rotary_prep(const RopePrepParams& p, cudaStream_t st) {
  if (p.seg[0].tokens == 0 && p.seg[1].tokens == 0) return ATTN_OK;
  return launch_rope_prep(p, st) == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

// The fp16 V pre-pass and the forward kernel, both on `stream`.  With a
// rotary, the V pre-pass launch also writes the rotated queries and keys
// (rp; tq and tk then describe those copies), in extra rows of blocks.
int launch_forward(const attn_shape* shape, const MaskParams& mask, const LayoutParams& lay, float scale,
                   const CUtensorMap& tq, const CUtensorMap& tk, const void* V, const FwdWorkspace& w, void* O,
                   float* LSE, void* O_lo, const RopePrepParams* rp, unsigned int* status, cudaStream_t st) {
  CUtensorMap tv;
  if (!make_tmap(&tv, w.V16, shape->d_v, w.nkt * kTileN, static_cast<int64_t>(shape->B) * shape->Hkv))
    return ATTN_ERR_CUDA;
  V16Params vp;
  vp.sh = shape_params(shape);
  vp.mask = mask;
  vp.lay = lay;
  vp.nkt = w.nkt;
  vp.V = V;
  vp.V16 = w.V16;
  vp.vexp = w.vexp;
  vp.status = status;
  vp.prep_rows = 0;
  std::memset(&vp.rp, 0, sizeof(vp.rp));
  if (rp) {
    // About two work items per prep thread, spread over whole rows of
    // B Hkv blocks.
    const int64_t items = (rp->seg[0].tokens + rp->seg[1].tokens) * (rp->d / 8);   // key rows (segment 0)
    const int64_t per_row = static_cast<int64_t>(shape->B) * shape->Hkv * 256 * 2;
    vp.prep_rows = static_cast<int32_t>(std::min<int64_t>(std::max<int64_t>((items + per_row - 1) / per_row, 1),
                                                          1024));
    vp.rp = *rp;
  }
  if (launch_attn_v16(shape->d_v, vp, st) != cudaSuccess) return ATTN_ERR_CUDA;
  FwdParams p;
  p.sh = vp.sh;
  p.mask = mask;
  p.lay = lay;
  p.scale_log2 = scale * kLog2e;
  p.wait_limit_ns = kDefaultWaitLimitNs;
  p.O = O;
  p.O_lo = O_lo;
  p.LSE = LSE;
  p.vexp = w.vexp;
  p.nkt = w.nkt;
  p.status = status;
  return launch_attn_fwd(shape->d_h, shape->d_v, tq, tk, tv, p, st) == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

int check_workspace(const attn_shape* s, const attn_rotary* r, const void* ws, size_t bytes) {
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return ATTN_ERR_WORKSPACE;
  if (bytes < workspace_layout(s, nullptr, r).bytes) return ATTN_ERR_WORKSPACE;
  return ATTN_OK;
}

__global__ void selftest_wait_kernel(uint64_t limit_ns, unsigned int* status) {
  __shared__ __align__(8) uint64_t never;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&never), 1);
    fence_mbar_init();
    abort_flag = 0;
  }
  __syncthreads();
  // Nothing ever arrives on this barrier: the wait has to give up by itself.
  const bool ok = mbar_wait(smem_u32(&never), 0, &abort_flag, limit_ns);
  if (!ok && threadIdx.x == 0) record_status(status, ATTN_ERR_TIMEOUT);
}

}  // namespace

// ---------------------------------------------------------------------------
// Static backward scratch for callers that cannot allocate device memory.
//
// The array is part of the library's device image: every GPU on which the
// library is loaded holds these bytes until the process exits.  In host code
// the name `g_static_bwd_scratch` is only a host-side stand-in for the
// symbol, never a device address, so it is never handed to a kernel; the
// device address comes from cudaGetSymbolAddress, looked up once per device
// (with that device current) on the first attn_bwd_noalloc call there.
// ---------------------------------------------------------------------------
constexpr size_t kStaticBwdScratchBytes = size_t{16} << 20;   // 16 MiB
static __device__ __align__(256) unsigned char g_static_bwd_scratch[kStaticBwdScratchBytes];

namespace {
std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxDevices] = {};

int static_scratch_ptr(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return ATTN_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return ATTN_ERR_DEVICE;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_static_bwd_scratch) != cudaSuccess || ptr == nullptr) return ATTN_ERR_CUDA;
    g_scratch_ptr[dev] = ptr;
  }
  *out = g_scratch_ptr[dev];
  return ATTN_OK;
}
// Layout of the short-query forward: query heads packed per 128-row tile,
// and the key range split so that the row tiles fill about two CTAs per SM.
struct DecodePlan {
  int heads_per_tile, chunks, nsplit;
  size_t opart_bytes, bytes;   // workspace: range outputs | range log-sum-exps
};

DecodePlan decode_plan(const attn_shape* s, const MaskParams& m) {
  constexpr int kTargetCtas = 2 * 152;
  const int group = s->Hq / s->Hkv;
  DecodePlan d;
  d.heads_per_tile = std::min(group, std::max(1, 128 / s->n_q));
  d.chunks = (group + d.heads_per_tile - 1) / d.heads_per_tile;
  const int64_t row_tiles = static_cast<int64_t>(s->B) * s->Hkv * d.chunks;
  int64_t max_tiles = 0;
  for (int b = 0; b < s->B; ++b) {
    const int64_t lim = row_key_limit(m, s->n_k, b, static_cast<int64_t>(s->n_q) - 1);
    max_tiles = std::max<int64_t>(max_tiles, (lim + kTileN - 1) / kTileN);
  }
  int64_t ns = (kTargetCtas + row_tiles - 1) / row_tiles;
  ns = std::min<int64_t>(ns, std::max<int64_t>(1, max_tiles / 2));   // at least two key tiles per range
  ns = std::min<int64_t>(std::max<int64_t>(ns, 1), 64);
  d.nsplit = static_cast<int>(ns);
  const size_t rows = static_cast<size_t>(s->B) * s->Hq * s->n_q;
  d.opart_bytes = d.nsplit > 1 ? round256(static_cast<size_t>(d.nsplit) * rows * s->d_v * sizeof(float)) : 0;
  d.bytes = d.nsplit > 1 ? d.opart_bytes + round256(static_cast<size_t>(d.nsplit) * rows * sizeof(float)) : 0;
  return d;
}

int check_decode_shape(const attn_shape* shape) {
  int rc = check_shape(shape);
  if (rc) return rc;
  return shape->n_q > 128 ? ATTN_ERR_UNSUPPORTED : ATTN_OK;
}

int check_rope(int64_t tokens, int32_t d, float base, const int32_t* positions, int32_t inverse) {
  if (tokens <= 0 || d <= 0 || d % 8 != 0 || d > 128) return ATTN_ERR_SHAPE;
  if (inverse != 0 && inverse != 1) return ATTN_ERR_SHAPE;
  if (!std::isfinite(base) || !(base > 1.f)) return ATTN_ERR_SCALE;
  if (!positions) return ATTN_ERR_NULL;
  return ATTN_OK;
}

int rope_launch(int64_t tokens, int32_t heads_a, int32_t heads_b, int32_t d, float base,
                const int32_t* positions, int32_t inverse, const void* Xa, void* Ya, const void* Xb, void* Yb,
                void* stream) {
  unsigned int* status = nullptr;
  int rc = device_status_ptr(&status);
  if (rc) return rc;
  float w_hi[64], w_lo[64];
  rope_frequencies(base, d, w_hi, w_lo);
  const cudaError_t e = launch_rope(tokens, d, heads_a, heads_b, positions, w_hi, w_lo, inverse, Xa, Ya, Xb, Yb,
                                    static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

}  // namespace
}  // namespace esd

using namespace esd;

extern "C" {

int attn_abi_version(void) { return ATTN_ABI_VERSION; }

const char* attn_strerror(int status) {
  switch (status) {
    case ATTN_OK: return "ok";
    case ATTN_ERR_NULL: return "a required pointer is NULL";
    case ATTN_ERR_SHAPE: return "invalid shape or mask parameters";
    case ATTN_ERR_UNSUPPORTED: return "unsupported head widths (d_h, d_v)";
    case ATTN_ERR_ALIGN: return "a tensor pointer is not 16-byte aligned";
    case ATTN_ERR_EMPTY_ROW: return "a query row has an empty visible set";
    case ATTN_ERR_SCALE: return "scale must be finite and > 0";
    case ATTN_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case ATTN_ERR_CUDA: return "a CUDA call or kernel launch failed";
    case ATTN_ERR_TIMEOUT: return "a kernel's bounded wait ran out";
    case ATTN_ERR_DEVICE: return "the current device is not an sm_103 GPU";
    case ATTN_ERR_RANGE: return "an input tile's magnitude (2^46 or more) was beyond the fp16 operands";
    default: return "unknown status";
  }
}

int attn_bwd_head_split(const attn_shape* shape, const attn_mask* mask) {
  if (check_shape(shape) != ATTN_OK) return -ATTN_ERR_SHAPE;
  MaskParams m;
  const int rc = build_mask(shape, mask, &m);
  if (rc) return -rc;
  unsigned int* status = nullptr;
  const int dc = device_status_ptr(&status);
  if (dc) return -dc;
  return choose_bwd_plan(shape, m, device_sms(), false).hsplit;
}

int attn_bwd_persistent(const attn_shape* shape, const attn_mask* mask, const attn_rotary* rotary) {
  if (check_shape(shape) != ATTN_OK) return -ATTN_ERR_SHAPE;
  MaskParams m;
  const int rc = build_mask(shape, mask, &m);
  if (rc) return -rc;
  unsigned int* status = nullptr;
  const int dc = device_status_ptr(&status);
  if (dc) return -dc;
  return choose_bwd_plan(shape, m, device_sms(), rotary != nullptr).persistent ? 1 : 0;
}

int64_t attn_visible_pairs(const attn_shape* shape, const attn_mask* mask) {
  if (check_shape(shape) != ATTN_OK) return -1;
  MaskParams m;
  if (build_mask(shape, mask, &m) != ATTN_OK) return -1;
  int64_t total = 0;
  for (int b = 0; b < shape->B; ++b) total += pairs_one_batch(m, shape->n_q, shape->n_k, b);
  return total * shape->Hq;
}

size_t attn_bwd_workspace_bytes(const attn_shape* shape, const attn_rotary* rotary) {
  if (check_shape(shape) != ATTN_OK || check_rotary(rotary) != ATTN_OK) return 0;
  return workspace_layout(shape, nullptr, rotary).bytes;
}

size_t attn_fwd_workspace_bytes(const attn_shape* shape, const attn_rotary* rotary) {
  if (check_shape(shape) != ATTN_OK || check_rotary(rotary) != ATTN_OK) return 0;
  return fwd_workspace_layout(shape, nullptr, padded_tokens(shape, rotary)).bytes;
}

int attn_fwd(const attn_shape* shape, const attn_mask* mask, const attn_strides* strides, const attn_rotary* rotary,
             float scale, const void* Q, const void* K, const void* V, void* O, float* LSE, void* O_lo,
             void* workspace, size_t workspace_bytes, void* stream) {
  int rc = check_shape(shape);
  if (rc) return rc;
  MaskParams m;
  rc = build_mask(shape, mask, &m);
  if (rc) return rc;
  rc = check_scale(scale);
  if (rc) return rc;
  LayoutParams lay;
  std::memset(&lay, 0, sizeof(lay));
  rc = build_strides(strides, shape->Hq, shape->Hkv, shape->n_q, shape->n_k, shape->d_h, shape->d_v, &lay);
  if (rc) return rc;
  rc = check_rotary(rotary);
  if (rc) return rc;
  rc = check_ptrs({Q, K, V, O, LSE});
  if (rc) return rc;
  if (O_lo && !aligned16(O_lo)) return ATTN_ERR_ALIGN;
  const RotaryTokens rt = padded_tokens(shape, rotary);
  rc = check_fwd_workspace(shape, rt, workspace, workspace_bytes);
  if (rc) return rc;
  // ---- CUDA from here on ----
  unsigned int* status = nullptr;
  rc = device_status_ptr(&status);
  if (rc) return rc;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  const FwdWorkspace w = fwd_workspace_layout(shape, workspace, rt);
  RopePrepParams rp;
  const void* Qa = Q;
  const void* Ka = K;
  if (rotary) {
    Qa = rotary->q_rot ? rotary->q_rot : w.Qr;
    Ka = rotary->k_rot ? rotary->k_rot : w.Kr;
    rp = rotary_prep(rotary, shape->d_h, false,
                     rope_segment(rt.q, shape->n_q, shape->Hq, rotary->pos_q, Q, lay.sq, const_cast<void*>(Qa)),
                     rope_segment(rt.k, shape->n_k, shape->Hkv, rotary->pos_k, K, lay.sk, const_cast<void*>(Ka)));
  }
  CUtensorMap tq, tk;
  const int64_t bhq = static_cast<int64_t>(shape->B) * shape->Hq;
  const int64_t bhk = static_cast<int64_t>(shape->B) * shape->Hkv;
  const bool ok = rotary ? make_tmap(&tq, Qa, shape->d_h, shape->n_q, bhq) &&
                               make_tmap(&tk, Ka, shape->d_h, shape->n_k, bhk)
                         : make_tmap(&tq, Q, shape->d_h, shape->n_q, bhq, lay.sq.row, lay.sq.head) &&
                               make_tmap(&tk, K, shape->d_h, shape->n_k, bhk, lay.sk.row, lay.sk.head);
  if (!ok) return ATTN_ERR_CUDA;
  return launch_forward(shape, m, lay, scale, tq, tk, V, w, O, LSE, O_lo, rotary ? &rp : nullptr, status, st);
}

size_t attn_fwd_decode_workspace_bytes(const attn_shape* shape, const attn_mask* mask) {
  if (check_decode_shape(shape) != ATTN_OK) return 0;
  MaskParams m;
  if (build_mask(shape, mask, &m) != ATTN_OK) return 0;
  return decode_plan(shape, m).bytes;
}

int attn_fwd_decode(const attn_shape* shape, const attn_mask* mask, float scale, const void* Q, const void* K,
                    const void* V, void* O, float* LSE, void* O_lo, void* workspace, size_t workspace_bytes,
                    void* stream) {
  int rc = check_decode_shape(shape);
  if (rc) return rc;
  DecParams p;
  rc = build_mask(shape, mask, &p.mask);
  if (rc) return rc;
  rc = check_scale(scale);
  if (rc) return rc;
  rc = check_ptrs({Q, K, V, O, LSE});
  if (rc) return rc;
  if (O_lo && !aligned16(O_lo)) return ATTN_ERR_ALIGN;
  const DecodePlan plan = decode_plan(shape, p.mask);
  if (plan.bytes > 0 &&
      (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 || workspace_bytes < plan.bytes))
    return ATTN_ERR_WORKSPACE;
  // ---- CUDA from here on ----
  unsigned int* status = nullptr;
  rc = device_status_ptr(&status);
  if (rc) return rc;
  CUtensorMap tk, tv;
  const int64_t bhk = static_cast<int64_t>(shape->B) * shape->Hkv;
  if (!make_tmap(&tk, K, shape->d_h, shape->n_k, bhk) || !make_tmap(&tv, V, shape->d_v, shape->n_k, bhk))
    return ATTN_ERR_CUDA;
  p.sh = shape_params(shape);
  p.scale_log2 = scale * kLog2e;
  p.wait_limit_ns = kDefaultWaitLimitNs;
  p.Q = Q;
  p.O = O;
  p.O_lo = O_lo;
  p.LSE = LSE;
  p.Opart = plan.bytes > 0 ? static_cast<float*>(workspace) : nullptr;
  p.Lpart = plan.bytes > 0 ? reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + plan.opart_bytes) : nullptr;
  p.heads_per_tile = plan.heads_per_tile;
  p.chunks = plan.chunks;
  p.nsplit = plan.nsplit;
  p.status = status;
  // Longest key range first: a CTA's work is proportional to its batch's
  // key tiles, and dispatching the long ones first keeps short ones for the
  // tail (the longest-processing-time-first list schedule).
  {
    int64_t ntiles[ATTN_MAX_BATCH];
    int16_t order[ATTN_MAX_BATCH];
    for (int b = 0; b < shape->B; ++b) {
      const int64_t lim = row_key_limit(p.mask, shape->n_k, b, static_cast<int64_t>(shape->n_q) - 1);
      ntiles[b] = lim > 0 ? (lim + kTileN - 1) / kTileN : 0;
      order[b] = static_cast<int16_t>(b);
    }
    std::stable_sort(order, order + shape->B, [&ntiles](int16_t x, int16_t y) { return ntiles[x] > ntiles[y]; });
    std::memset(p.batch_order, 0, sizeof(p.batch_order));
    for (int b = 0; b < shape->B; ++b) p.batch_order[b] = order[b];
  }
  const cudaError_t e = launch_attn_decode(shape->d_h, shape->d_v, tk, tv, p, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

// Stage 1.  With a rotary, Q is turned as it is read, or the forward's
// rotated queries (q_rot) are read instead.
int attn_bwd_preprocess(const attn_shape* shape, const attn_strides* strides, const attn_rotary* rotary,
                        const void* Q, const void* O, const void* O_lo, const void* dO, void* workspace,
                        size_t workspace_bytes, void* stream) {
  int rc = check_shape(shape);
  if (rc) return rc;
  LayoutParams padded;
  std::memset(&padded, 0, sizeof(padded));
  rc = build_strides(strides, shape->Hq, shape->Hkv, shape->n_q, shape->n_k, shape->d_h, shape->d_v, &padded);
  if (rc) return rc;
  rc = check_rotary(rotary);
  if (rc) return rc;
  rc = check_ptrs({Q, O, O_lo, dO});
  if (rc) return rc;
  rc = check_workspace(shape, rotary, workspace, workspace_bytes);
  if (rc) return rc;
  unsigned int* status = nullptr;
  rc = device_status_ptr(&status);
  if (rc) return rc;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  const Workspace w = workspace_layout(shape, workspace, rotary);
  RotaryAngles ra;
  const bool turn = rotary && !rotary->q_rot;
  if (turn) ra = rotary_angles(rotary, rotary->pos_q, shape->d_h);
  if (rotary && rotary->q_rot) {
    Q = rotary->q_rot;   // contiguous rows
    padded.sq = TensorStrides{shape->d_h, static_cast<int64_t>(shape->n_q) * shape->d_h};
  }
  const cudaError_t e = launch_attn_bwd_preprocess(shape_params(shape), padded, shape->d_v, shape->d_h, Q, O, O_lo,
                                                   dO, w.D, w.tilemax, w.grpexp, w.work_ctr, w.dQacc, w.Q16,
                                                   w.dO16,
                                                   turn ? &ra : nullptr, status, st);
  return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

// Stage 2.  With a rotary, the keys are the forward's rotated keys (k_rot)
// or a rotated copy written into the workspace first; dK is turned back.
int attn_bwd_main(const attn_shape* shape, const attn_mask* mask, const attn_strides* strides,
                  const attn_rotary* rotary, float scale, const void* K, const void* V, const float* LSE,
                  void* workspace, size_t workspace_bytes, void* dK, void* dV, void* stream) {
  int rc = check_shape(shape);
  if (rc) return rc;
  BwdParams p;
  rc = build_mask(shape, mask, &p.mask);
  if (rc) return rc;
  std::memset(&p.lay, 0, sizeof(p.lay));
  rc = build_strides(strides, shape->Hq, shape->Hkv, shape->n_q, shape->n_k, shape->d_h, shape->d_v, &p.lay);
  if (rc) return rc;
  rc = check_scale(scale);
  if (rc) return rc;
  rc = check_rotary(rotary);
  if (rc) return rc;
  rc = check_ptrs({K, V, LSE, dK, dV});
  if (rc) return rc;
  rc = check_workspace(shape, rotary, workspace, workspace_bytes);
  if (rc) return rc;
  const Workspace w = workspace_layout(shape, workspace, rotary);
  unsigned int* status = nullptr;
  rc = device_status_ptr(&status);
  if (rc) return rc;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  const void* Ka = K;
  if (rotary) {
    Ka = rotary->k_rot ? rotary->k_rot : w.Kr;
    if (!rotary->k_rot) {
      const RotaryTokens rt = padded_tokens(shape, rotary);
      const RopeSegment none = rope_segment(0, 0, 0, nullptr, nullptr, TensorStrides{0, 0}, nullptr);
      rc = launch_rotary_prep(rotary_prep(rotary, shape->d_h, false,
                                          rope_segment(rt.k, shape->n_k, shape->Hkv, rotary->pos_k, K, p.lay.sk,
                                                       w.Kr),
                                          none),
                              st);
      if (rc) return rc;
    }
  }
  CUtensorMap tq, tk, tv, tdo, tdq;
  const int64_t bhq = static_cast<int64_t>(shape->B) * shape->Hq;
  const int64_t bhk = static_cast<int64_t>(shape->B) * shape->Hkv;
  const bool k_ok = rotary ? make_tmap(&tk, Ka, shape->d_h, shape->n_k, bhk)
                           : make_tmap(&tk, K, shape->d_h, shape->n_k, bhk, p.lay.sk.row, p.lay.sk.head);
  if (!make_tmap(&tq, w.Q16, shape->d_h, shape->n_q, bhq) || !k_ok ||
      !make_tmap(&tv, V, shape->d_v, shape->n_k, bhk, p.lay.sv.row, p.lay.sv.head) ||
      !make_tmap(&tdo, w.dO16, shape->d_v, shape->n_q, bhq) || !make_tmap_acc(&tdq, w.dQacc, shape->d_h, shape->n_q, bhq))
    return ATTN_ERR_CUDA;
  p.sh = shape_params(shape);
  p.scale = scale;
  p.scale_log2 = scale * kLog2e;
  p.wait_limit_ns = kDefaultWaitLimitNs;
  p.LSE = LSE;
  p.D = w.D;
  p.tilemax = w.tilemax;
  p.grpexp = w.grpexp;
  p.nqt = (shape->n_q + 127) / 128;
  p.dQacc = w.dQacc;
  p.dK = dK;
  p.dV = dV;
  if (rotary) p.rot = rotary_angles(rotary, rotary->pos_k, shape->d_h);
  else p.rot.pos = nullptr;
  p.status = status;
  const BwdPlan plan = choose_bwd_plan(shape, p.mask, device_sms(), rotary != nullptr);
  p.hsplit = plan.hsplit;
  p.persistent = plan.persistent ? 1 : 0;
  p.dKacc = w.dKacc;
  p.dVacc = w.dVacc;
  if (!set_bwd_schedule(&p, w, device_sms())) return ATTN_ERR_SHAPE;
  if (p.hsplit > 1 && launch_zero_f32(w.dKacc, static_cast<int64_t>(w.kv_elems), st) != cudaSuccess)
    return ATTN_ERR_CUDA;
  cudaError_t e = launch_attn_bwd_main(shape->d_h, shape->d_v, tq, tk, tv, tdo, tdq, p, st);
  if (e == cudaSuccess && p.hsplit > 1)
    e = launch_attn_bwd_kv_finalize(p.sh, p.lay, static_cast<int64_t>(shape->B) * shape->n_k, shape->d_h,
                                    shape->d_v, w.dKacc, w.dVacc, dK, dV, st);
  return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

int attn_bwd_finalize(const attn_shape* shape, const attn_strides* strides, const attn_rotary* rotary, float scale,
                      const void* workspace, size_t workspace_bytes, void* dQ, void* stream) {
  int rc = check_shape(shape);
  if (rc) return rc;
  LayoutParams lay;
  std::memset(&lay, 0, sizeof(lay));
  rc = build_strides(strides, shape->Hq, shape->Hkv, shape->n_q, shape->n_k, shape->d_h, shape->d_v, &lay);
  if (rc) return rc;
  rc = check_scale(scale);
  if (rc) return rc;
  rc = check_rotary(rotary);
  if (rc) return rc;
  rc = check_ptrs({dQ});
  if (rc) return rc;
  rc = check_workspace(shape, rotary, workspace, workspace_bytes);
  if (rc) return rc;
  unsigned int* status = nullptr;
  rc = device_status_ptr(&status);
  if (rc) return rc;
  const Workspace w = workspace_layout(shape, const_cast<void*>(workspace), rotary);
  RotaryAngles ra;
  if (rotary) ra = rotary_angles(rotary, rotary->pos_q, shape->d_h);
  // Padded accumulator rows: heads of n_q rows.
  const cudaError_t e = launch_attn_bwd_finalize(
      q_rows(shape) * shape->d_h, shape->d_h, shape->n_q, lay.sdq.head, lay.sdq.row,
      contiguous_strides(lay, lay.sdq, shape->Hq, shape->n_q, shape->d_h), scale, w.dQacc, dQ,
      rotary ? &ra : nullptr, false, shape->Hq, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

int attn_bwd(const attn_shape* shape, const attn_mask* mask, const attn_strides* strides, const attn_rotary* rotary,
             float scale, const void* Q, const void* K, const void* V, const void* O, const void* O_lo, const void* dO,
             const float* LSE, void* dQ, void* dK, void* dV, void* workspace, size_t workspace_bytes, void* stream) {
  int rc = check_shape(shape);
  if (rc) return rc;
  MaskParams m;
  rc = build_mask(shape, mask, &m);
  if (rc) return rc;
  {
    LayoutParams lay;
    std::memset(&lay, 0, sizeof(lay));
    rc = build_strides(strides, shape->Hq, shape->Hkv, shape->n_q, shape->n_k, shape->d_h, shape->d_v, &lay);
    if (rc) return rc;
  }
  rc = check_scale(scale);
  if (rc) return rc;
  rc = check_rotary(rotary);
  if (rc) return rc;
  rc = check_ptrs({Q, K, V, O, O_lo, dO, LSE, dQ, dK, dV});
  if (rc) return rc;
  rc = check_workspace(shape, rotary, workspace, workspace_bytes);
  if (rc) return rc;
  rc = attn_bwd_preprocess(shape, strides, rotary, Q, O, O_lo, dO, workspace, workspace_bytes, stream);
  if (rc) return rc;
  rc = attn_bwd_main(shape, mask, strides, rotary, scale, K, V, LSE, workspace, workspace_bytes, dK, dV, stream);
  if (rc) return rc;
  return attn_bwd_finalize(shape, strides, rotary, scale, workspace, workspace_bytes, dQ, stream);
}

int attn_get_status(int* status) {
  if (!status) return ATTN_ERR_NULL;
  unsigned int* dev_status = nullptr;
  const int rc = device_status_ptr(&dev_status);
  if (rc) return rc;
  unsigned int v = 0;
  if (cudaDeviceSynchronize() != cudaSuccess) return ATTN_ERR_CUDA;
  if (cudaMemcpy(&v, dev_status, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return ATTN_ERR_CUDA;
  *status = static_cast<int>(v);
  return ATTN_OK;
}

int attn_clear_status(void) {
  unsigned int* dev_status = nullptr;
  const int rc = device_status_ptr(&dev_status);
  if (rc) return rc;
  if (cudaDeviceSynchronize() != cudaSuccess) return ATTN_ERR_CUDA;
  const unsigned int zero = 0;
  if (cudaMemcpy(dev_status, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess) return ATTN_ERR_CUDA;
  return ATTN_OK;
}

int attn_selftest_wait_timeout(uint64_t limit_ns, void* stream) {
  unsigned int* dev_status = nullptr;
  const int rc = device_status_ptr(&dev_status);
  if (rc) return rc;
  selftest_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(limit_ns, dev_status);
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

// The backward pass for callers that cannot call cudaMalloc: identical to
// attn_bwd, but its scratch is the library's static device buffer instead of
// a caller workspace.  Problems whose scratch would exceed the buffer are
// refused with ATTN_ERR_WORKSPACE before anything is launched.  The stage
// kernels rewrite every byte they read back (the dQ accumulator is zeroed by
// the preprocess stage), so leftovers from an earlier call do not matter; but
// all calls share the one buffer, so calls that overlap on the GPU (other
// streams, other host threads) race and must be serialised by the caller.
int attn_bwd_noalloc(const attn_shape* shape, const attn_mask* mask, const attn_strides* strides,
                     const attn_rotary* rotary, float scale, const void* Q, const void* K, const void* V,
                     const void* O, const void* O_lo, const void* dO, const float* LSE, void* dQ, void* dK, void* dV,
                     void* stream) {
  int rc = check_shape(shape);
  if (rc) return rc;
  rc = check_rotary(rotary);
  if (rc) return rc;
  if (workspace_layout(shape, nullptr, rotary).bytes > kStaticBwdScratchBytes) return ATTN_ERR_WORKSPACE;
  // Every argument check before the first CUDA call (the symbol lookup).
  MaskParams m;
  rc = build_mask(shape, mask, &m);
  if (rc) return rc;
  {
    LayoutParams lay;
    std::memset(&lay, 0, sizeof(lay));
    rc = build_strides(strides, shape->Hq, shape->Hkv, shape->n_q, shape->n_k, shape->d_h, shape->d_v, &lay);
    if (rc) return rc;
  }
  rc = check_scale(scale);
  if (rc) return rc;
  rc = check_ptrs({Q, K, V, O, O_lo, dO, LSE, dQ, dK, dV});
  if (rc) return rc;
  void* scratch = nullptr;
  rc = static_scratch_ptr(&scratch);
  if (rc) return rc;
  return attn_bwd(shape, mask, strides, rotary, scale, Q, K, V, O, O_lo, dO, LSE, dQ, dK, dV, scratch,
                  kStaticBwdScratchBytes, stream);
}

size_t attn_bwd_noalloc_max_scratch_bytes(void) { return kStaticBwdScratchBytes; }

// ---------------------------------------------------------------------------
// Projections on either side of attention (A.10.10-A.10.11)
// ---------------------------------------------------------------------------
int attn_rope(int64_t tokens, int32_t heads, int32_t d, float base, const int32_t* positions, int32_t inverse,
              const void* X, void* Y, void* stream) {
  if (heads <= 0) return ATTN_ERR_SHAPE;
  int rc = check_rope(tokens, d, base, positions, inverse);
  if (rc) return rc;
  rc = check_ptrs({X, Y});
  if (rc) return rc;
  return rope_launch(tokens, heads, 0, d, base, positions, inverse, X, Y, nullptr, nullptr, stream);
}

int attn_rope_qk(int64_t tokens, int32_t heads_q, int32_t heads_k, int32_t d, float base,
                 const int32_t* positions, int32_t inverse, const void* Xq, void* Yq, const void* Xk, void* Yk,
                 void* stream) {
  if (heads_q <= 0 || heads_k <= 0) return ATTN_ERR_SHAPE;
  int rc = check_rope(tokens, d, base, positions, inverse);
  if (rc) return rc;
  rc = check_ptrs({Xq, Yq, Xk, Yk});
  if (rc) return rc;
  return rope_launch(tokens, heads_q, heads_k, d, base, positions, inverse, Xq, Yq, Xk, Yk, stream);
}

int attn_proj_fwd(int64_t T, int32_t D, int32_t N, const void* X, const void* W, void* Y, void* stream) {
  int rc = check_proj_dims(T, D, N);
  if (rc) return rc;
  rc = check_ptrs({X, W, Y});
  if (rc) return rc;
  unsigned int* status = nullptr;
  rc = device_status_ptr(&status);
  if (rc) return rc;
  CUtensorMap tA[3], tB[3];
  // A = X [T][D] K-major (boxes 64 x 128), B = W [D][N] MN-major (boxes 64 x 64).
  if (!make_tmap_2d(&tA[0], X, T, D, 64, 128) || !make_tmap_2d(&tB[0], W, D, N, 64, 64)) return ATTN_ERR_CUDA;
  tA[1] = tA[2] = tA[0];
  tB[1] = tB[2] = tB[0];
  GemmParams p{};
  p.M = T;
  p.N = N;
  p.nsrc = 1;
  p.K[0] = D;
  p.ldc = N;
  p.C = Y;
  p.wait_limit_ns = kDefaultWaitLimitNs;
  p.status = status;
  return launch_proj_gemm(kGemmXW, tA, tB, p, static_cast<cudaStream_t>(stream)) == cudaSuccess ? ATTN_OK
                                                                                                : ATTN_ERR_CUDA;
}

int attn_proj_bwd_weight(int64_t T, int32_t D, int32_t N, const void* X, const void* G, float* dW, void* stream) {
  int rc = check_proj_dims(T, D, N);
  if (rc) return rc;
  rc = check_ptrs({X, G, dW});
  if (rc) return rc;
  unsigned int* status = nullptr;
  rc = device_status_ptr(&status);
  if (rc) return rc;
  CUtensorMap tA[3], tB[3];
  // A = X^T: X [T][D] read MN-major (boxes 64 x 64); B = G [T][N] MN-major.
  if (!make_tmap_2d(&tA[0], X, T, D, 64, 64) || !make_tmap_2d(&tB[0], G, T, N, 64, 64)) return ATTN_ERR_CUDA;
  tA[1] = tA[2] = tA[0];
  tB[1] = tB[2] = tB[0];
  GemmParams p{};
  p.M = D;
  p.N = N;
  p.nsrc = 1;
  p.K[0] = static_cast<int32_t>(T);
  p.ldc = N;
  p.C = dW;
  p.wait_limit_ns = kDefaultWaitLimitNs;
  p.status = status;
  return launch_proj_gemm(kGemmXtG, tA, tB, p, static_cast<cudaStream_t>(stream)) == cudaSuccess ? ATTN_OK
                                                                                                 : ATTN_ERR_CUDA;
}

int attn_proj_bwd_input(int64_t T, int32_t D, int32_t nsrc, const int32_t* N, const void* const* G,
                        const void* const* W, void* dX, void* stream) {
  if (!N || !G || !W) return ATTN_ERR_NULL;
  if (nsrc < 1 || nsrc > 3) return ATTN_ERR_SHAPE;
  int rc = ATTN_OK;
  for (int s = 0; s < nsrc; ++s) {
    rc = check_proj_dims(T, D, N[s]);
    if (rc) return rc;
    rc = check_ptrs({G[s], W[s]});
    if (rc) return rc;
  }
  rc = check_ptrs({dX});
  if (rc) return rc;
  unsigned int* status = nullptr;
  rc = device_status_ptr(&status);
  if (rc) return rc;
  CUtensorMap tA[3], tB[3];
  GemmParams p{};
  for (int s = 0; s < 3; ++s) {
    const int k = s < nsrc ? s : 0;
    // A = G_s [T][N_s] K-major (boxes 64 x 128); B = W_s^T: W_s [D][N_s] K-major (boxes 64 x 256).
    if (!make_tmap_2d(&tA[s], G[k], T, N[k], 64, 128) || !make_tmap_2d(&tB[s], W[k], D, N[k], 64, 256))
      return ATTN_ERR_CUDA;
    p.K[s] = s < nsrc ? N[s] : 0;
  }
  p.M = T;
  p.N = D;
  p.nsrc = nsrc;
  p.ldc = D;
  p.C = dX;
  p.wait_limit_ns = kDefaultWaitLimitNs;
  p.status = status;
  return launch_proj_gemm(kGemmGWt, tA, tB, p, static_cast<cudaStream_t>(stream)) == cudaSuccess ? ATTN_OK
                                                                                                 : ATTN_ERR_CUDA;
}

// ---------------------------------------------------------------------------
// Packed variable-length sequences: the same kernels, addressing rows through
// the token offsets (LayoutParams) and the per-sequence lengths (MaskParams).
// ---------------------------------------------------------------------------
int64_t attn_varlen_visible_pairs(const attn_varlen* v) {
  Varlen d;
  if (build_varlen(v, &d) != ATTN_OK) return -1;
  int64_t total = 0;
  for (int b = 0; b < v->B; ++b) total += pairs_one_batch(d.mask, d.shape.n_q, d.shape.n_k, b);
  return total * v->Hq;
}

size_t attn_fwd_varlen_workspace_bytes(const attn_varlen* v, const attn_rotary* rotary) {
  Varlen d;
  if (build_varlen(v, &d) != ATTN_OK || check_rotary(rotary) != ATTN_OK) return 0;
  return fwd_workspace_layout(&d.shape, nullptr, varlen_tokens(d, rotary)).bytes;
}

int attn_fwd_varlen(const attn_varlen* v, const attn_strides* strides, const attn_rotary* rotary, float scale,
                    const void* Q, const void* K, const void* V, void* O, float* LSE, void* O_lo, void* workspace,
                    size_t workspace_bytes, void* stream) {
  Varlen d;
  int rc = build_varlen(v, &d);
  if (rc) return rc;
  rc = build_strides(strides, v->Hq, v->Hkv, 0, 0, v->d_h, v->d_v, &d.lay);
  if (rc) return rc;
  rc = check_scale(scale);
  if (rc) return rc;
  rc = check_rotary(rotary);
  if (rc) return rc;
  if (d.total_q == 0) return ATTN_OK;   // no query rows: nothing to write
  rc = check_ptrs({Q, K, V, O, LSE});
  if (rc) return rc;
  if (O_lo && !aligned16(O_lo)) return ATTN_ERR_ALIGN;
  const RotaryTokens rt = varlen_tokens(d, rotary);
  rc = check_fwd_workspace(&d.shape, rt, workspace, workspace_bytes);
  if (rc) return rc;
  // ---- CUDA from here on ----
  unsigned int* status = nullptr;
  rc = device_status_ptr(&status);
  if (rc) return rc;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  const FwdWorkspace w = fwd_workspace_layout(&d.shape, workspace, rt);
  RopePrepParams rp;
  const void* Qa = Q;
  const void* Ka = K;
  if (rotary) {
    Qa = rotary->q_rot ? rotary->q_rot : w.Qr;
    Ka = rotary->k_rot ? rotary->k_rot : w.Kr;
    rp = rotary_prep(rotary, v->d_h, true,
                     rope_segment(rt.q, 0, v->Hq, rotary->pos_q, Q, d.lay.sq, const_cast<void*>(Qa)),
                     rope_segment(rt.k, 0, v->Hkv, rotary->pos_k, K, d.lay.sk, const_cast<void*>(Ka)));
  }
  CUtensorMap tq, tk;
  const bool ok = rotary ? make_tmap_packed(&tq, Qa, v->d_h, v->Hq, d.total_q) &&
                               make_tmap_packed(&tk, Ka, v->d_h, v->Hkv, d.total_k)
                         : make_tmap_packed(&tq, Q, v->d_h, v->Hq, d.total_q, d.lay.sq.row, d.lay.sq.head) &&
                               make_tmap_packed(&tk, K, v->d_h, v->Hkv, d.total_k, d.lay.sk.row, d.lay.sk.head);
  if (!ok) return ATTN_ERR_CUDA;
  return launch_forward(&d.shape, d.mask, d.lay, scale, tq, tk, V, w, O, LSE, O_lo, rotary ? &rp : nullptr, status,
                        st);
}

size_t attn_bwd_varlen_workspace_bytes(const attn_varlen* v, const attn_rotary* rotary) {
  Varlen d;
  if (build_varlen(v, &d) != ATTN_OK || check_rotary(rotary) != ATTN_OK) return 0;
  return workspace_layout_varlen(d, nullptr, rotary).bytes;
}

int attn_bwd_varlen(const attn_varlen* v, const attn_strides* strides, const attn_rotary* rotary, float scale,
                    const void* Q, const void* K, const void* V, const void* O, const void* O_lo, const void* dO,
                    const float* LSE, void* dQ, void* dK, void* dV, void* workspace, size_t workspace_bytes,
                    void* stream) {
  Varlen d;
  int rc = build_varlen(v, &d);
  if (rc) return rc;
  rc = build_strides(strides, v->Hq, v->Hkv, 0, 0, v->d_h, v->d_v, &d.lay);
  if (rc) return rc;
  rc = check_scale(scale);
  if (rc) return rc;
  rc = check_rotary(rotary);
  if (rc) return rc;
  if (d.total_k > 0) {
    rc = check_ptrs({K, V, dK, dV});
    if (rc) return rc;
  }
  if (d.total_q > 0) {
    rc = check_ptrs({Q, O, O_lo, dO, LSE, dQ});
    if (rc) return rc;
    const Workspace need = workspace_layout_varlen(d, nullptr, rotary);
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 || workspace_bytes < need.bytes)
      return ATTN_ERR_WORKSPACE;
  }
  // ---- CUDA from here on ----
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (d.total_k == 0) return ATTN_OK;
  if (d.total_q == 0) {
    // No query sees any key: the gradients of K and V are zero (each head's
    // rows as one pitched block: tokens at the row stride, d elements each).
    auto zero = [&](void* t, const TensorStrides& s, int d_) {
      for (int h = 0; h < v->Hkv; ++h)
        if (cudaMemset2DAsync(static_cast<__nv_bfloat16*>(t) + static_cast<int64_t>(h) * s.head,
                              static_cast<size_t>(s.row) * 2, 0, static_cast<size_t>(d_) * 2,
                              static_cast<size_t>(d.total_k), st) != cudaSuccess)
          return false;
      return true;
    };
    if (!zero(dK, d.lay.sdk, v->d_h) || !zero(dV, d.lay.sdv, v->d_v)) return ATTN_ERR_CUDA;
    return ATTN_OK;
  }
  unsigned int* status = nullptr;
  rc = device_status_ptr(&status);
  if (rc) return rc;
  const Workspace w = workspace_layout_varlen(d, workspace, rotary);
  const ShapeParams sh = shape_params(&d.shape);
  if (rotary) {
    // The rotated keys, unless the forward's are given.
    if (!rotary->k_rot) {
      const RopeSegment none = rope_segment(0, 0, 0, nullptr, nullptr, TensorStrides{0, 0}, nullptr);
      rc = launch_rotary_prep(
          rotary_prep(rotary, v->d_h, true, rope_segment(d.total_k, 0, v->Hkv, rotary->pos_k, K, d.lay.sk, w.Kr),
                      none),
          st);
      if (rc) return rc;
    }
  }
  RotaryAngles rq, rk;
  LayoutParams play = d.lay;   // the preprocess's view of Q
  const void* Qa = Q;
  const bool turn_q = rotary && !rotary->q_rot;
  if (rotary) {
    rq = rotary_angles(rotary, rotary->pos_q, v->d_h);
    rk = rotary_angles(rotary, rotary->pos_k, v->d_h);
    if (rotary->q_rot) {
      Qa = rotary->q_rot;
      play.sq = TensorStrides{static_cast<int64_t>(v->Hq) * v->d_h, v->d_h};
    }
  }
  cudaError_t e = launch_attn_bwd_preprocess(sh, play, v->d_v, v->d_h, Qa, O, O_lo, dO, w.D, w.tilemax, w.grpexp,
                                             w.work_ctr, w.dQacc, w.Q16, w.dO16, turn_q ? &rq : nullptr, status, st);
  if (e != cudaSuccess) return ATTN_ERR_CUDA;
  CUtensorMap tq, tk, tv, tdo, tdq;
  const bool k_ok =
      rotary ? make_tmap_packed(&tk, rotary->k_rot ? rotary->k_rot : w.Kr, v->d_h, v->Hkv, d.total_k)
             : make_tmap_packed(&tk, K, v->d_h, v->Hkv, d.total_k, d.lay.sk.row, d.lay.sk.head);
  if (!make_tmap_packed(&tq, w.Q16, v->d_h, v->Hq, d.total_q) || !k_ok ||
      !make_tmap_packed(&tv, V, v->d_v, v->Hkv, d.total_k, d.lay.sv.row, d.lay.sv.head) ||
      !make_tmap_packed(&tdo, w.dO16, v->d_v, v->Hq, d.total_q) ||
      !make_tmap_acc_packed(&tdq, w.dQacc, v->d_h, v->Hq, d.total_q))
    return ATTN_ERR_CUDA;
  BwdParams p;
  p.sh = sh;
  p.mask = d.mask;
  p.lay = d.lay;
  p.scale = scale;
  p.scale_log2 = scale * kLog2e;
  p.wait_limit_ns = kDefaultWaitLimitNs;
  p.LSE = LSE;
  p.D = w.D;
  p.tilemax = w.tilemax;
  p.grpexp = w.grpexp;
  p.nqt = (d.shape.n_q + 127) / 128;
  p.dQacc = w.dQacc;
  p.dK = dK;
  p.dV = dV;
  if (rotary) p.rot = rk;
  else p.rot.pos = nullptr;
  p.status = status;
  const BwdPlan plan = choose_bwd_plan(&d.shape, d.mask, device_sms(), rotary != nullptr);
  p.hsplit = plan.hsplit;
  p.persistent = plan.persistent ? 1 : 0;
  p.dKacc = w.dKacc;
  p.dVacc = w.dVacc;
  if (!set_bwd_schedule(&p, w, device_sms())) return ATTN_ERR_SHAPE;
  if (p.hsplit > 1 && launch_zero_f32(w.dKacc, static_cast<int64_t>(w.kv_elems), st) != cudaSuccess)
    return ATTN_ERR_CUDA;
  e = launch_attn_bwd_main(v->d_h, v->d_v, tq, tk, tv, tdo, tdq, p, st);
  if (e == cudaSuccess && p.hsplit > 1)
    e = launch_attn_bwd_kv_finalize(sh, d.lay, d.total_k, v->d_h, v->d_v, w.dKacc, w.dVacc, dK, dV, st);
  if (e != cudaSuccess) return ATTN_ERR_CUDA;
  // Packed accumulator rows: tokens of Hq heads.
  e = launch_attn_bwd_finalize(d.total_q * v->Hq * v->d_h, v->d_h, v->Hq, d.lay.sdq.row, d.lay.sdq.head,
                               contiguous_strides(d.lay, d.lay.sdq, v->Hq, 0, v->d_h), scale, w.dQacc, dQ,
                               rotary ? &rq : nullptr, true, v->Hq, st);
  return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

}  // extern "C"
