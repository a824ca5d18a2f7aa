// C ABI of the attention library (declared in include/fa_gb300.h):
// argument validation, TMA tensor-map construction, device status word, and
// dispatch to the kernel translation units.  No allocation happens here.
#include <cudaTypedefs.h>
#include <math.h>
#include <stdint.h>

#include "../../include/fa_gb300.h"
#include "fa_decode.h"
#include "fa_internal.h"

namespace {

// Device status block: kernels OR fa::kStatus* bits into word 0 and add to the
// score-block counters behind it (layout in fa_internal.h).
__device__ __align__(16) unsigned int g_fa_status[fa::kStatusWords];

unsigned int* status_word() {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_fa_status) != cudaSuccess) return nullptr;
  return static_cast<unsigned int*>(p);
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = []() -> PFN_cuTensorMapEncodeTiled_v12000 {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }();
  return fn;
}

bool aligned16(const void* p) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

constexpr float kLog2e = 1.4426950408889634f;

fa_status check_scale(float scale) {
  return (isfinite(scale) && scale > 0.f) ? FA_OK : FA_ERR_INVALID_ARG;
}

// One attention problem as the kernels see it: head dimension, dtype and the
// row layout (dense [B, H, N, d] or packed variable-length [T, H, d]).
struct Shape {
  int B = 0, H = 0, d = 0, dtype = 0;
  fa::SeqLayout lay;
  bool varlen() const { return lay.cu_q != nullptr; }
  long long q_rows() const { return varlen() ? (long long)lay.Tq * H : (long long)B * H * lay.Nq; }
  bool bf16() const { return dtype == FA_BF16; }
  int width() const { return d == 64 ? 64 : d == 256 ? 256 : 128; }  // compute width (96 runs at 128)
};

fa_status check_dims(int d, int dtype) {
  if (dtype != FA_FP16 && dtype != FA_BF16) return FA_ERR_UNSUPPORTED;
  if (d != 64 && d != 96 && d != 128 && d != 256) return FA_ERR_UNSUPPORTED;
  return FA_OK;
}

fa_status dense_shape(int B, int H, int Nq, int Nk, int d, int dtype, Shape* s) {
  if (B < 1 || H < 1 || Nq < 1 || Nk < 1) return FA_ERR_INVALID_ARG;
  const fa_status st = check_dims(d, dtype);
  if (st != FA_OK) return st;
  const long long BH = (long long)B * H;
  if (BH * Nq * d >= (1LL << 31) || BH * Nk * d >= (1LL << 31)) return FA_ERR_UNSUPPORTED;
  s->B = B;
  s->H = H;
  s->d = d;
  s->dtype = dtype;
  s->lay = fa::SeqLayout();
  s->lay.H = H;
  s->lay.Nq = Nq;
  s->lay.Nk = Nk;
  s->lay.dh = d;
  return FA_OK;
}

fa_status varlen_shape(const int* cu_q, const int* cu_k, int B, int H, int max_q, int max_k, int total_q,
                       int total_k, int d, int dtype, Shape* s) {
  if (!cu_q || !cu_k || (reinterpret_cast<uintptr_t>(cu_q) & 3u) || (reinterpret_cast<uintptr_t>(cu_k) & 3u))
    return FA_ERR_INVALID_ARG;
  if (B < 1 || H < 1 || max_q < 1 || max_k < 1 || total_q < 1 || total_k < 1) return FA_ERR_INVALID_ARG;
  const fa_status st = check_dims(d, dtype);
  if (st != FA_OK) return st;
  if ((long long)total_q * H * d >= (1LL << 31) || (long long)total_k * H * d >= (1LL << 31))
    return FA_ERR_UNSUPPORTED;
  s->B = B;
  s->H = H;
  s->d = d;
  s->dtype = dtype;
  s->lay = fa::SeqLayout();
  s->lay.cu_q = cu_q;
  s->lay.cu_k = cu_k;
  s->lay.H = H;
  s->lay.Nq = max_q;
  s->lay.Nk = max_k;
  s->lay.Tq = total_q;
  s->lay.Tk = total_k;
  s->lay.dh = d;
  return FA_OK;
}

// 3-D tiled TMA map over the query-side (key_side = false) or key-side rows
// of `s`: boxes of 64 columns x `box_rows` rows, 128-byte swizzle; rows and
// columns out of range read as 0 (d = 96: columns 96-127 of the second box).
//   dense:  dims (d, N, B*H), box {64, box_rows, 1}
//   varlen: dims (d, H, T),   box {64, 1, box_rows}  (strides increase)
bool make_map(CUtensorMap* m, const void* ptr, const Shape& s, bool key_side, int box_rows) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t d = (cuuint64_t)s.d;
  cuuint64_t dims[3];
  cuuint64_t strides[2];
  cuuint32_t box[3];
  if (s.varlen()) {
    const cuuint64_t T = (cuuint64_t)(key_side ? s.lay.Tk : s.lay.Tq);
    dims[0] = d;
    dims[1] = (cuuint64_t)s.H;
    dims[2] = T;
    strides[0] = d * 2;
    strides[1] = (cuuint64_t)s.H * d * 2;
    box[0] = 64;
    box[1] = 1;
    box[2] = (cuuint32_t)box_rows;
  } else {
    const cuuint64_t N = (cuuint64_t)(key_side ? s.lay.Nk : s.lay.Nq);
    dims[0] = d;
    dims[1] = N;
    dims[2] = (cuuint64_t)s.B * s.H;
    strides[0] = d * 2;
    strides[1] = N * d * 2;
    box[0] = 64;
    box[1] = (cuuint32_t)box_rows;
    box[2] = 1;
  }
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(m, s.bf16() ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
                   const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Dropout probability -> generator parameters: t = round(p * 256), keep
// scale 256 / (256 - t).  False for p outside [0, 1) (NaN included) or p
// rounding to 1.
bool make_drop(float p, uint64_t seed, uint32_t offset, fa::DropParams* dp) {
  if (!(p >= 0.f && p < 1.f)) return false;
  const double t = floor((double)p * 256.0 + 0.5);
  if (t >= 256.0) return false;
  dp->t = (uint32_t)t;
  dp->keep_scale = (float)(256.0 / (256.0 - t));
  dp->k0 = (uint32_t)(seed & 0xffffffffu);
  dp->k1 = (uint32_t)(seed >> 32);
  dp->offset = offset;
  return true;
}

fa_status check_block_mask(const uint8_t* block_mask, int mask_heads, int B, int H) {
  if (!block_mask) return FA_ERR_INVALID_ARG;
  if (mask_heads != 1 && (long long)mask_heads != (long long)B * H) return FA_ERR_INVALID_ARG;
  return FA_OK;
}

// ---------------------------------------------------------------- runners
fa_status run_forward(const Shape& s, const void* q, const void* k, const void* v, void* o, float* lse,
                      const uint8_t* block_mask, int mask_heads, int causal, float scale, void* stream,
                      const fa::DropParams* drop) {
  fa_status st = check_scale(scale);
  if (st != FA_OK) return st;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
    return FA_ERR_INVALID_ARG;
  if (s.d == 256 && block_mask) return FA_ERR_UNSUPPORTED;
  fa::FwdArgs a;
  if (!make_map(&a.tm_q, q, s, false, 128) || !make_map(&a.tm_k, k, s, true, 128) ||
      !make_map(&a.tm_v, v, s, true, 128) || !make_map(&a.tm_o, o, s, false, 128))
    return FA_ERR_CUDA;
  a.o = o;
  a.lse = lse;
  a.lay = s.lay;
  a.BH = s.B * s.H;
  a.scale_log2 = scale * kLog2e;
  a.block_mask = block_mask;
  a.mask_heads = mask_heads;
  a.status = status_word();
  if (!a.status) return FA_ERR_CUDA;
  // p rounding to 0 drops nothing: the plain kernel computes exactly that.
  a.dropout = drop != nullptr && drop->t > 0;
  if (a.dropout) a.drop = *drop;
  const cudaStream_t cs = static_cast<cudaStream_t>(stream);
  const cudaError_t e = s.d == 256   ? fa::launch_forward256(causal != 0, s.bf16(), a, cs)
                        : s.varlen()  ? fa::launch_forward_varlen(s.width(), causal != 0, s.bf16(), a, cs)
                        : a.dropout ? fa::launch_forward_dropout(s.width(), causal != 0, s.bf16(), a, cs)
                                    : fa::launch_forward(s.width(), causal != 0, s.bf16(), a, cs);
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

// dq_accum may be null: then only D is computed (the split backward needs no accumulator).
fa_status run_preprocess(const Shape& s, const void* o, const void* dO, float* delta, float* dq_accum,
                         void* stream) {
  if (!aligned16(o) || !aligned16(dO) || !aligned16(delta) || (dq_accum && !aligned16(dq_accum)))
    return FA_ERR_INVALID_ARG;
  if (fa::launch_backward_preprocess(s.d, s.bf16(), o, dO, delta, dq_accum, s.q_rows(),
                                     static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return FA_ERR_CUDA;
  return FA_OK;
}

fa_status run_dkdv(const Shape& s, const void* q, const void* k, const void* v, const void* dO, const float* lse,
                   const float* delta, float* dq_accum, void* dk, void* dv, const uint8_t* block_mask,
                   int mask_heads, int causal, float scale, void* stream, const fa::DropParams* drop) {
  fa_status st = check_scale(scale);
  if (st != FA_OK) return st;
  if (s.d == 256 && block_mask) return FA_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(dO) || !aligned16(lse) ||
      !aligned16(delta) || !aligned16(dq_accum) || !aligned16(dk) || !aligned16(dv))
    return FA_ERR_INVALID_ARG;
  const int bq = fa::backward_q_tile(s.width());
  fa::BwdArgs a;
  if (!make_map(&a.tm_q, q, s, false, bq) || !make_map(&a.tm_do, dO, s, false, bq) ||
      !make_map(&a.tm_k, k, s, true, 128) || !make_map(&a.tm_v, v, s, true, 128) ||
      !make_map(&a.tm_dk, dk, s, true, 128) || !make_map(&a.tm_dv, dv, s, true, 128))
    return FA_ERR_CUDA;
  a.dk = dk;
  a.dv = dv;
  a.lse = lse;
  a.delta = delta;
  a.dq_accum = dq_accum;
  a.lay = s.lay;
  a.BH = s.B * s.H;
  a.scale = scale;
  a.scale_log2 = scale * kLog2e;
  a.block_mask = block_mask;
  a.mask_heads = mask_heads;
  a.status = status_word();
  if (!a.status) return FA_ERR_CUDA;
  a.dropout = drop != nullptr && drop->t > 0;
  if (a.dropout) a.drop = *drop;
  const cudaStream_t cs = static_cast<cudaStream_t>(stream);
  const cudaError_t e = s.varlen()  ? fa::launch_backward_dkdv_varlen(s.width(), causal != 0, s.bf16(), a, cs)
                        : a.dropout ? fa::launch_backward_dkdv_dropout(s.width(), causal != 0, s.bf16(), a, cs)
                                    : fa::launch_backward_dkdv(s.width(), causal != 0, s.bf16(), a, cs);
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

// The two stages of the split backward: dK and dV (want_dq false) or dQ
// (want_dq true), each recomputing P and dP; d in {64, 96, 128}; dense
// layouts with a block mask or with dropout (not both), or packed layouts
// without dropout.
fa_status run_split(const Shape& s, bool want_dq, const void* q, const void* k, const void* v, const void* dO,
                    const float* lse, const float* delta, void* dq, void* dk, void* dv, const uint8_t* block_mask,
                    int mask_heads, int causal, float scale, void* stream, const fa::DropParams* drop = nullptr) {
  fa_status st = check_scale(scale);
  if (st != FA_OK) return st;
  const bool dropping = drop != nullptr && drop->t > 0;
  if (s.width() == 256 || (dropping && (s.varlen() || block_mask))) return FA_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(dO) || !aligned16(lse) || !aligned16(delta))
    return FA_ERR_INVALID_ARG;
  if (want_dq ? !aligned16(dq) : (!aligned16(dk) || !aligned16(dv))) return FA_ERR_INVALID_ARG;
  fa::SplitArgs a;
  if (!make_map(&a.tm_q, q, s, false, 128) || !make_map(&a.tm_do, dO, s, false, 128) ||
      !make_map(&a.tm_k, k, s, true, 128) || !make_map(&a.tm_v, v, s, true, 128))
    return FA_ERR_CUDA;
  if (!want_dq && (!make_map(&a.tm_dk, dk, s, true, 128) || !make_map(&a.tm_dv, dv, s, true, 128)))
    return FA_ERR_CUDA;
  a.dq = dq;
  a.dk = dk;
  a.dv = dv;
  a.lse = lse;
  a.delta = delta;
  a.lay = s.lay;
  a.BH = s.B * s.H;
  a.dh = s.d;
  a.scale = scale;
  a.scale_log2 = scale * kLog2e;
  a.block_mask = block_mask;
  a.mask_heads = mask_heads;
  a.dropout = dropping;
  if (dropping) a.drop = *drop;
  a.status = status_word();
  if (!a.status) return FA_ERR_CUDA;
  const cudaStream_t cs = static_cast<cudaStream_t>(stream);
  const cudaError_t e = want_dq ? fa::launch_backward_dq(s.width(), causal != 0, s.bf16(), a, cs)
                                : fa::launch_backward_dkdv_split(s.width(), causal != 0, s.bf16(), a, cs);
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

fa_status run_convert(const Shape& s, const float* dq_accum, void* dq, float scale, void* stream) {
  fa_status st = check_scale(scale);
  if (st != FA_OK) return st;
  if (!aligned16(dq_accum) || !aligned16(dq)) return FA_ERR_INVALID_ARG;
  if (fa::launch_backward_dq_convert(s.d, s.bf16(), dq_accum, dq, s.q_rows(), scale,
                                     static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return FA_ERR_CUDA;
  return FA_OK;
}

size_t workspace_bytes_for(const Shape& s) {
  const size_t rows = (size_t)s.q_rows();
  return align256(rows * sizeof(float)) + align256(rows * s.d * sizeof(float));
}

// Everything run_backward checks except the workspace: scale, head dim with a
// block mask, and every tensor pointer (non-null, 16-byte aligned).
fa_status check_backward(const Shape& s, const void* q, const void* k, const void* v, const void* o, const void* dO,
                         const float* lse, const void* dq, const void* dk, const void* dv, const uint8_t* block_mask,
                         float scale) {
  fa_status st = check_scale(scale);
  if (st != FA_OK) return st;
  if (s.d == 256 && block_mask) return FA_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(dO) || !aligned16(lse) ||
      !aligned16(dq) || !aligned16(dk) || !aligned16(dv))
    return FA_ERR_INVALID_ARG;
  return FA_OK;
}

fa_status run_backward(const Shape& s, const void* q, const void* k, const void* v, const void* o, const void* dO,
                       const float* lse, void* dq, void* dk, void* dv, const uint8_t* block_mask, int mask_heads,
                       int causal, float scale, void* workspace, size_t workspace_bytes, void* stream,
                       const fa::DropParams* drop) {
  // Every argument is checked here, before the first of the three launches.
  fa_status st = check_backward(s, q, k, v, o, dO, lse, dq, dk, dv, block_mask, scale);
  if (st != FA_OK) return st;
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) || workspace_bytes < workspace_bytes_for(s))
    return FA_ERR_WORKSPACE;
  float* delta = static_cast<float*>(workspace);
  float* dq_accum =
      reinterpret_cast<float*>(static_cast<char*>(workspace) + align256((size_t)s.q_rows() * sizeof(float)));
  // d <= 128 without dropout (dense with or without a block mask, or packed)
  // takes the split backward (dQ by its own kernel, no accumulator); d = 256
  // and dropout accumulate dQ in the dK / dV kernel.  With dropout the split
  // kernels would each draw the keep mask again on their softmax warps'
  // critical path (C4, p = 0.1: 2.90 + 1.66 ms against 3.51 ms for the
  // accumulating kernel, whose otherwise idle dQ-drain warps draw it once).
  const bool split = s.width() != 256 && !(drop && drop->t > 0);
  if (split) {
    if ((st = run_preprocess(s, o, dO, delta, nullptr, stream)) != FA_OK) return st;
    if ((st = run_split(s, false, q, k, v, dO, lse, delta, nullptr, dk, dv, block_mask, mask_heads, causal, scale,
                        stream, drop)) != FA_OK)
      return st;
    return run_split(s, true, q, k, v, dO, lse, delta, dq, nullptr, nullptr, block_mask, mask_heads, causal, scale,
                     stream, drop);
  }
  if ((st = run_preprocess(s, o, dO, delta, dq_accum, stream)) != FA_OK) return st;
  if ((st = run_dkdv(s, q, k, v, dO, lse, delta, dq_accum, dk, dv, block_mask, mask_heads, causal, scale, stream,
                     drop)) != FA_OK)
    return st;
  return run_convert(s, dq_accum, dq, scale, stream);
}

}  // namespace

namespace fa {
int backward_arguments_status(const void* q, const void* k, const void* v, const void* o, const void* dO,
                              const float* lse, const void* dq, const void* dk, const void* dv, int B, int H, int N,
                              int d, int dtype, float scale) {
  Shape s;
  const fa_status st = dense_shape(B, H, N, N, d, dtype, &s);
  if (st != FA_OK) return st;
  return check_backward(s, q, k, v, o, dO, lse, dq, dk, dv, nullptr, scale);
}
}  // namespace fa

// ---------------------------------------------------------------- entry points
extern "C" {

const char* fa_status_string(int status) {
  switch (status) {
    case FA_OK: return "FA_OK";
    case FA_ERR_INVALID_ARG: return "FA_ERR_INVALID_ARG: null/misaligned pointer, bad size or bad scale";
    case FA_ERR_UNSUPPORTED:
      return "FA_ERR_UNSUPPORTED: head dim must be 64, 96, 128 or 256 (no block mask at 256), dtype fp16/bf16, "
             "rows*H*d < 2^31";
    case FA_ERR_CUDA: return "FA_ERR_CUDA: a CUDA launch or the stream failed";
    case FA_ERR_TIMEOUT: return "FA_ERR_TIMEOUT: a kernel gave up waiting on its pipeline";
    case FA_ERR_WORKSPACE: return "FA_ERR_WORKSPACE: workspace missing, misaligned or too small";
    case FA_ERR_SCRATCH_TOO_SMALL:
      return "FA_ERR_SCRATCH_TOO_SMALL: fa_backward_noalloc needs more than its fixed 32 MiB scratch; use fa_backward";
    case FA_ERR_SEQLENS:
      return "FA_ERR_SEQLENS: a cu_seqlens range exceeded the packed totals or the maximum lengths; it was skipped";
    default: return "unknown fa_status";
  }
}

fa_status fa_forward(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N,
                     int d, int dtype, int causal, float scale, void* stream) {
  Shape s;
  const fa_status st = dense_shape(B, H, N, N, d, dtype, &s);
  if (st != FA_OK) return st;
  return run_forward(s, q, k, v, o, lse, nullptr, 1, causal, scale, stream, nullptr);
}

fa_status fa_forward_blocksparse(const void* q, const void* k, const void* v, void* o, float* lse,
                                 const uint8_t* block_mask, int mask_heads, int B, int H, int N, int d, int dtype,
                                 int causal, float scale, void* stream) {
  Shape s;
  fa_status st = dense_shape(B, H, N, N, d, dtype, &s);
  if (st != FA_OK) return st;
  if ((st = check_block_mask(block_mask, mask_heads, B, H)) != FA_OK) return st;
  return run_forward(s, q, k, v, o, lse, block_mask, mask_heads, causal, scale, stream, nullptr);
}

fa_status fa_forward_dropout(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N,
                             int d, int dtype, int causal, float scale, float p_drop, uint64_t seed,
                             uint32_t offset, void* stream) {
  Shape s;
  const fa_status st = dense_shape(B, H, N, N, d, dtype, &s);
  if (st != FA_OK) return st;
  fa::DropParams dp;
  if (!make_drop(p_drop, seed, offset, &dp)) return FA_ERR_INVALID_ARG;
  return run_forward(s, q, k, v, o, lse, nullptr, 1, causal, scale, stream, &dp);
}

fa_status fa_forward_varlen(const void* q, const void* k, const void* v, void* o, float* lse, const int* cu_seqlens_q,
                            const int* cu_seqlens_k, int B, int H, int max_seqlen_q, int max_seqlen_k, int total_q,
                            int total_k, int d, int dtype, int causal, float scale, float p_drop, uint64_t seed,
                            uint32_t offset, void* stream) {
  Shape s;
  const fa_status st = varlen_shape(cu_seqlens_q, cu_seqlens_k, B, H, max_seqlen_q, max_seqlen_k, total_q, total_k,
                                    d, dtype, &s);
  if (st != FA_OK) return st;
  fa::DropParams dp;
  if (!make_drop(p_drop, seed, offset, &dp)) return FA_ERR_INVALID_ARG;
  return run_forward(s, q, k, v, o, lse, nullptr, 1, causal, scale, stream, &dp);
}

size_t fa_backward_workspace_size(int B, int H, int N, int d) {
  Shape s;
  if (dense_shape(B, H, N, N, d, FA_BF16, &s) != FA_OK) return 0;
  return workspace_bytes_for(s);
}

size_t fa_backward_varlen_workspace_size(int total_q, int H, int d) {
  if (total_q < 1 || H < 1 || check_dims(d, FA_BF16) != FA_OK) return 0;
  if ((long long)total_q * H * d >= (1LL << 31)) return 0;
  const size_t rows = (size_t)total_q * H;
  return align256(rows * sizeof(float)) + align256(rows * d * sizeof(float));
}

fa_status fa_backward(const void* q, const void* k, const void* v, const void* o, const void* dO,
                      const float* lse, void* dq, void* dk, void* dv, int B, int H, int N, int d, int dtype,
                      int causal, float scale, void* workspace, size_t workspace_bytes, void* stream) {
  Shape s;
  const fa_status st = dense_shape(B, H, N, N, d, dtype, &s);
  if (st != FA_OK) return st;
  return run_backward(s, q, k, v, o, dO, lse, dq, dk, dv, nullptr, 1, causal, scale, workspace, workspace_bytes,
                      stream, nullptr);
}

fa_status fa_backward_blocksparse(const void* q, const void* k, const void* v, const void* o, const void* dO,
                                  const float* lse, void* dq, void* dk, void* dv, const uint8_t* block_mask,
                                  int mask_heads, int B, int H, int N, int d, int dtype, int causal, float scale,
                                  void* workspace, size_t workspace_bytes, void* stream) {
  Shape s;
  fa_status st = dense_shape(B, H, N, N, d, dtype, &s);
  if (st != FA_OK) return st;
  if ((st = check_block_mask(block_mask, mask_heads, B, H)) != FA_OK) return st;
  return run_backward(s, q, k, v, o, dO, lse, dq, dk, dv, block_mask, mask_heads, causal, scale, workspace,
                      workspace_bytes, stream, nullptr);
}

fa_status fa_backward_dropout(const void* q, const void* k, const void* v, const void* o, const void* dO,
                              const float* lse, void* dq, void* dk, void* dv, int B, int H, int N, int d, int dtype,
                              int causal, float scale, float p_drop, uint64_t seed, uint32_t offset, void* workspace,
                              size_t workspace_bytes, void* stream) {
  Shape s;
  const fa_status st = dense_shape(B, H, N, N, d, dtype, &s);
  if (st != FA_OK) return st;
  fa::DropParams dp;
  if (!make_drop(p_drop, seed, offset, &dp)) return FA_ERR_INVALID_ARG;
  return run_backward(s, q, k, v, o, dO, lse, dq, dk, dv, nullptr, 1, causal, scale, workspace, workspace_bytes,
                      stream, &dp);
}

fa_status fa_backward_varlen(const void* q, const void* k, const void* v, const void* o, const void* dO,
                             const float* lse, void* dq, void* dk, void* dv, const int* cu_seqlens_q,
                             const int* cu_seqlens_k, int B, int H, int max_seqlen_q, int max_seqlen_k, int total_q,
                             int total_k, int d, int dtype, int causal, float scale, float p_drop, uint64_t seed,
                             uint32_t offset, void* workspace, size_t workspace_bytes, void* stream) {
  Shape s;
  const fa_status st = varlen_shape(cu_seqlens_q, cu_seqlens_k, B, H, max_seqlen_q, max_seqlen_k, total_q, total_k,
                                    d, dtype, &s);
  if (st != FA_OK) return st;
  fa::DropParams dp;
  if (!make_drop(p_drop, seed, offset, &dp)) return FA_ERR_INVALID_ARG;
  return run_backward(s, q, k, v, o, dO, lse, dq, dk, dv, nullptr, 1, causal, scale, workspace, workspace_bytes,
                      stream, &dp);
}

fa_status fa_backward_dkdv_varlen(const void* q, const void* k, const void* v, const void* dO, const float* lse,
                                  const float* delta, float* dq_accum, void* dk, void* dv, const int* cu_seqlens_q,
                                  const int* cu_seqlens_k, int B, int H, int max_seqlen_q, int max_seqlen_k,
                                  int total_q, int total_k, int d, int dtype, int causal, float scale, float p_drop,
                                  uint64_t seed, uint32_t offset, void* stream) {
  Shape s;
  const fa_status st = varlen_shape(cu_seqlens_q, cu_seqlens_k, B, H, max_seqlen_q, max_seqlen_k, total_q, total_k,
                                    d, dtype, &s);
  if (st != FA_OK) return st;
  fa::DropParams dp;
  if (!make_drop(p_drop, seed, offset, &dp)) return FA_ERR_INVALID_ARG;
  return run_dkdv(s, q, k, v, dO, lse, delta, dq_accum, dk, dv, nullptr, 1, causal, scale, stream, &dp);
}

fa_status fa_backward_dk_dv_varlen(const void* q, const void* k, const void* v, const void* dO, const float* lse,
                                  const float* delta, void* dk, void* dv, const int* cu_seqlens_q,
                                  const int* cu_seqlens_k, int B, int H, int max_seqlen_q, int max_seqlen_k,
                                  int total_q, int total_k, int d, int dtype, int causal, float scale, void* stream) {
  Shape s;
  const fa_status st = varlen_shape(cu_seqlens_q, cu_seqlens_k, B, H, max_seqlen_q, max_seqlen_k, total_q, total_k,
                                    d, dtype, &s);
  if (st != FA_OK) return st;
  return run_split(s, false, q, k, v, dO, lse, delta, nullptr, dk, dv, nullptr, 1, causal, scale, stream);
}

fa_status fa_backward_dq_varlen(const void* q, const void* k, const void* v, const void* dO, const float* lse,
                                const float* delta, void* dq, const int* cu_seqlens_q, const int* cu_seqlens_k, int B,
                                int H, int max_seqlen_q, int max_seqlen_k, int total_q, int total_k, int d, int dtype,
                                int causal, float scale, void* stream) {
  Shape s;
  const fa_status st = varlen_shape(cu_seqlens_q, cu_seqlens_k, B, H, max_seqlen_q, max_seqlen_k, total_q, total_k,
                                    d, dtype, &s);
  if (st != FA_OK) return st;
  return run_split(s, true, q, k, v, dO, lse, delta, dq, nullptr, nullptr, nullptr, 1, causal, scale, stream);
}

fa_status fa_backward_preprocess(const void* o, const void* dO, float* delta, float* dq_accum, int B, int H,
                                 int N, int d, int dtype, void* stream) {
  Shape s;
  const fa_status st = dense_shape(B, H, N, N, d, dtype, &s);
  if (st != FA_OK) return st;
  return run_preprocess(s, o, dO, delta, dq_accum, stream);
}

fa_status fa_backward_dkdv(const void* q, const void* k, const void* v, const void* dO, const float* lse,
                           const float* delta, float* dq_accum, void* dk, void* dv, int B, int H, int N, int d,
                           int dtype, int causal, float scale, void* stream) {
  Shape s;
  const fa_status st = dense_shape(B, H, N, N, d, dtype, &s);
  if (st != FA_OK) return st;
  return run_dkdv(s, q, k, v, dO, lse, delta, dq_accum, dk, dv, nullptr, 1, causal, scale, stream, nullptr);
}

fa_status fa_backward_dkdv_blocksparse(const void* q, const void* k, const void* v, const void* dO, const float* lse,
                                       const float* delta, float* dq_accum, void* dk, void* dv,
                                       const uint8_t* block_mask, int mask_heads, int B, int H, int N, int d,
                                       int dtype, int causal, float scale, void* stream) {
  Shape s;
  fa_status st = dense_shape(B, H, N, N, d, dtype, &s);
  if (st != FA_OK) return st;
  if ((st = check_block_mask(block_mask, mask_heads, B, H)) != FA_OK) return st;
  return run_dkdv(s, q, k, v, dO, lse, delta, dq_accum, dk, dv, block_mask, mask_heads, causal, scale, stream,
                  nullptr);
}

fa_status fa_backward_dkdv_dropout(const void* q, const void* k, const void* v, const void* dO, const float* lse,
                                   const float* delta, float* dq_accum, void* dk, void* dv, int B, int H, int N,
                                   int d, int dtype, int causal, float scale, float p_drop, uint64_t seed,
                                   uint32_t offset, void* stream) {
  Shape s;
  const fa_status st = dense_shape(B, H, N, N, d, dtype, &s);
  if (st != FA_OK) return st;
  fa::DropParams dp;
  if (!make_drop(p_drop, seed, offset, &dp)) return FA_ERR_INVALID_ARG;
  return run_dkdv(s, q, k, v, dO, lse, delta, dq_accum, dk, dv, nullptr, 1, causal, scale, stream, &dp);
}

fa_status fa_backward_dk_dv(const void* q, const void* k, const void* v, const void* dO, const float* lse,
                            const float* delta, void* dk, void* dv, int B, int H, int N, int d, int dtype, int causal,
                            float scale, void* stream) {
  Shape s;
  const fa_status st = dense_shape(B, H, N, N, d, dtype, &s);
  if (st != FA_OK) return st;
  return run_split(s, false, q, k, v, dO, lse, delta, nullptr, dk, dv, nullptr, 1, causal, scale, stream);
}

fa_status fa_backward_dq(const void* q, const void* k, const void* v, const void* dO, const float* lse,
                         const float* delta, void* dq, int B, int H, int N, int d, int dtype, int causal, float scale,
                         void* stream) {
  Shape s;
  const fa_status st = dense_shape(B, H, N, N, d, dtype, &s);
  if (st != FA_OK) return st;
  return run_split(s, true, q, k, v, dO, lse, delta, dq, nullptr, nullptr, nullptr, 1, causal, scale, stream);
}

fa_status fa_backward_dk_dv_blocksparse(const void* q, const void* k, const void* v, const void* dO,
                                        const float* lse, const float* delta, void* dk, void* dv,
                                        const uint8_t* block_mask, int mask_heads, int B, int H, int N, int d,
                                        int dtype, int causal, float scale, void* stream) {
  Shape s;
  fa_status st = dense_shape(B, H, N, N, d, dtype, &s);
  if (st != FA_OK) return st;
  if ((st = check_block_mask(block_mask, mask_heads, B, H)) != FA_OK) return st;
  return run_split(s, false, q, k, v, dO, lse, delta, nullptr, dk, dv, block_mask, mask_heads, causal, scale, stream);
}

fa_status fa_backward_dq_blocksparse(const void* q, const void* k, const void* v, const void* dO, const float* lse,
                                     const float* delta, void* dq, const uint8_t* block_mask, int mask_heads, int B,
                                     int H, int N, int d, int dtype, int causal, float scale, void* stream) {
  Shape s;
  fa_status st = dense_shape(B, H, N, N, d, dtype, &s);
  if (st != FA_OK) return st;
  if ((st = check_block_mask(block_mask, mask_heads, B, H)) != FA_OK) return st;
  return run_split(s, true, q, k, v, dO, lse, delta, dq, nullptr, nullptr, block_mask, mask_heads, causal, scale,
                   stream);
}

fa_status fa_backward_dk_dv_dropout(const void* q, const void* k, const void* v, const void* dO, const float* lse,
                                    const float* delta, void* dk, void* dv, int B, int H, int N, int d, int dtype,
                                    int causal, float scale, float p_drop, uint64_t seed, uint32_t offset,
                                    void* stream) {
  Shape s;
  const fa_status st = dense_shape(B, H, N, N, d, dtype, &s);
  if (st != FA_OK) return st;
  fa::DropParams dp;
  if (!make_drop(p_drop, seed, offset, &dp)) return FA_ERR_INVALID_ARG;
  return run_split(s, false, q, k, v, dO, lse, delta, nullptr, dk, dv, nullptr, 1, causal, scale, stream, &dp);
}

fa_status fa_backward_dq_dropout(const void* q, const void* k, const void* v, const void* dO, const float* lse,
                                 const float* delta, void* dq, int B, int H, int N, int d, int dtype, int causal,
                                 float scale, float p_drop, uint64_t seed, uint32_t offset, void* stream) {
  Shape s;
  const fa_status st = dense_shape(B, H, N, N, d, dtype, &s);
  if (st != FA_OK) return st;
  fa::DropParams dp;
  if (!make_drop(p_drop, seed, offset, &dp)) return FA_ERR_INVALID_ARG;
  return run_split(s, true, q, k, v, dO, lse, delta, dq, nullptr, nullptr, nullptr, 1, causal, scale, stream, &dp);
}

fa_status fa_backward_dq_convert(const float* dq_accum, void* dq, int B, int H, int N, int d, int dtype,
                                 float scale, void* stream) {
  Shape s;
  const fa_status st = dense_shape(B, H, N, N, d, dtype, &s);
  if (st != FA_OK) return st;
  return run_convert(s, dq_accum, dq, scale, stream);
}

fa_status fa_dropout_keep_mask(uint8_t* keep, int BH, int Nq, int Nk, float p_drop, uint64_t seed, uint32_t offset,
                               void* stream) {
  fa::DropParams dp;
  if (!make_drop(p_drop, seed, offset, &dp)) return FA_ERR_INVALID_ARG;
  if (BH < 1 || Nq < 1 || Nk < 1 || !keep) return FA_ERR_INVALID_ARG;
  if (fa::launch_dropout_keep_mask(keep, BH, Nq, Nk, dp, static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return FA_ERR_CUDA;
  return FA_OK;
}

}  // extern "C"

// ---------------------------------------------------------------- decoding
namespace {

// Query rows of one K / V head when Hq query heads share Hkv K / V heads.
fa_status gqa_rows(int Hq, int Hkv, int Nq, int* rows) {
  if (Hq < 1 || Hkv < 1 || Nq < 1 || Hq % Hkv != 0) return FA_ERR_INVALID_ARG;
  const long long r = (long long)(Hq / Hkv) * Nq;
  if (r > 0x7fffffffLL) return FA_ERR_UNSUPPORTED;
  *rows = (int)r;
  return FA_OK;
}

fa_status decode_plan(int B, int H, int Nq, int Nk, int d, int num_splits, int* splits, int* chunk,
                      size_t* bytes) {
  if (B < 1 || H < 1 || Nq < 1 || Nk < 1) return FA_ERR_INVALID_ARG;
  if (d != 64 && d != 128 && d != 256) return FA_ERR_UNSUPPORTED;
  const long long BH = (long long)B * H;
  if (BH > 65535 || BH * Nk * d >= (1LL << 31) || BH * Nq * d >= (1LL << 31)) return FA_ERR_UNSUPPORTED;
  if (num_splits < 0 || num_splits > 1024) return FA_ERR_INVALID_ARG;
  int s = num_splits ? num_splits : fa::decode_default_splits((int)BH, Nq, Nk);
  const int c = fa::decode_chunk(Nk, s);
  s = (Nk + c - 1) / c;  // no empty trailing chunk
  const size_t rows = (size_t)s * BH * Nq;
  *splits = s;
  *chunk = c;
  *bytes = align256(rows * d * sizeof(float)) + align256(rows * sizeof(float));
  return FA_OK;
}

}  // namespace

extern "C" {

size_t fa_decode_workspace_size(int B, int H, int Nq, int Nk, int d, int num_splits) {
  int s, c;
  size_t bytes = 0;
  return decode_plan(B, H, Nq, Nk, d, num_splits, &s, &c, &bytes) == FA_OK ? bytes : 0;
}

fa_status fa_forward_decode(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                            int Nq, int Nk, int d, int dtype, int causal, float scale, int num_splits,
                            void* workspace, size_t workspace_bytes, void* stream) {
  return fa_forward_decode_gqa(q, k, v, o, lse, B, H, H, Nq, Nk, d, dtype, causal, scale, num_splits, workspace,
                               workspace_bytes, stream);
}

size_t fa_decode_gqa_workspace_size(int B, int Hq, int Hkv, int Nq, int Nk, int d, int num_splits) {
  int rows;
  if (gqa_rows(Hq, Hkv, Nq, &rows) != FA_OK) return 0;
  int s, c;
  size_t bytes = 0;
  return decode_plan(B, Hkv, rows, Nk, d, num_splits, &s, &c, &bytes) == FA_OK ? bytes : 0;
}

fa_status fa_forward_decode_gqa(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq,
                                int Hkv, int Nq, int Nk, int d, int dtype, int causal, float scale, int num_splits,
                                void* workspace, size_t workspace_bytes, void* stream) {
  // The Hq / Hkv query heads of a K / V head are consecutive in q, o and lse,
  // so they form one block of rows = (Hq / Hkv) * Nq query rows of that head.
  int rows;
  fa_status st = gqa_rows(Hq, Hkv, Nq, &rows);
  if (st != FA_OK) return st;
  int splits, chunk;
  size_t need;
  if ((st = decode_plan(B, Hkv, rows, Nk, d, num_splits, &splits, &chunk, &need)) != FA_OK) return st;
  if (dtype != FA_FP16 && dtype != FA_BF16) return FA_ERR_UNSUPPORTED;
  if ((st = check_scale(scale)) != FA_OK) return st;
  if (causal && Nq > Nk) return FA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
    return FA_ERR_INVALID_ARG;
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) || workspace_bytes < need)
    return FA_ERR_WORKSPACE;
  fa::DecodeArgs a;
  a.o = o;
  a.lse = lse;
  a.BH = B * Hkv;
  a.Nq = rows;
  a.Nk = Nk;
  a.num_splits = splits;
  a.chunk = chunk;
  a.causal = causal != 0;
  a.scale_log2 = scale * kLog2e;
  const size_t part_rows = (size_t)splits * a.BH * rows;
  a.o_part = static_cast<float*>(workspace);
  a.lse_part = reinterpret_cast<float*>(static_cast<char*>(workspace) + align256(part_rows * d * sizeof(float)));
  const cudaStream_t cs = static_cast<cudaStream_t>(stream);
  Shape sh;  // q viewed as [B, Hkv, rows, d], k and v as [B, Hkv, Nk, d]
  if (dense_shape(B, Hkv, rows, Nk, d, dtype, &sh) != FA_OK) return FA_ERR_INVALID_ARG;
  if (!make_map(&a.tm_q, q, sh, false, 128) || !make_map(&a.tm_k, k, sh, true, 128) ||
      !make_map(&a.tm_v, v, sh, true, 128))
    return FA_ERR_CUDA;
  a.status = status_word();
  if (!a.status) return FA_ERR_CUDA;
  if (fa::launch_decode_tc_grouped(d, dtype == FA_BF16, a, Nq, cs) != cudaSuccess) return FA_ERR_CUDA;
  return fa::launch_decode_combine(d, dtype == FA_BF16, a, cs) == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

fa_status fa_selftest_wait_timeout(void* stream) {
  unsigned int* st = status_word();
  if (!st) return FA_ERR_CUDA;
  if (fa::launch_selftest_wait_timeout(st, static_cast<cudaStream_t>(stream)) != cudaSuccess) return FA_ERR_CUDA;
  return FA_OK;
}

fa_status fa_device_status(void* stream) {
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return FA_ERR_CUDA;
  unsigned int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_fa_status, sizeof(v)) != cudaSuccess) return FA_ERR_CUDA;
  if (v != 0) {
    const unsigned int zero = 0;
    if (cudaMemcpyToSymbol(g_fa_status, &zero, sizeof(zero)) != cudaSuccess) return FA_ERR_CUDA;
    if (v & fa::kStatusTimeout) return FA_ERR_TIMEOUT;
    if (v & fa::kStatusBadSeqlens) return FA_ERR_SEQLENS;
  }
  return FA_OK;
}

fa_status fa_score_blocks(void* stream, unsigned long long* fwd_blocks, unsigned long long* bwd_blocks, int reset) {
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return FA_ERR_CUDA;
  unsigned long long c[2] = {0ull, 0ull};
  if (cudaMemcpyFromSymbol(c, g_fa_status, sizeof(c), 2 * sizeof(unsigned int)) != cudaSuccess) return FA_ERR_CUDA;
  if (fwd_blocks) *fwd_blocks = c[fa::kCountForward];
  if (bwd_blocks) *bwd_blocks = c[fa::kCountBackward];
  if (reset) {
    const unsigned long long zero[2] = {0ull, 0ull};
    if (cudaMemcpyToSymbol(g_fa_status, zero, sizeof(zero), 2 * sizeof(unsigned int)) != cudaSuccess)
      return FA_ERR_CUDA;
  }
  return FA_OK;
}

}  // extern "C"
