// C ABI of the attention library (declared in include/fa_gb300.h):
// argument validation, TMA tensor-map construction, device status word, and
// dispatch to the kernel translation units.  No allocation happens here.
#include <cudaTypedefs.h>
#include <math.h>
#include <stdint.h>

#include "../../include/fa_gb300.h"
#include "fa_internal.h"

namespace {

// Device status word: kernels OR fa::kStatus* bits into it.
__device__ unsigned int g_fa_status;

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

// 3-D tiled map over a contiguous [BH, N, d] 16-bit tensor: box of 64 columns
// x `box_rows` rows x 1 head, 128-byte swizzle, out-of-range rows read as 0.
bool make_map(CUtensorMap* m, const void* ptr, bool bf16, int d, int N, int BH, int box_rows) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)N, (cuuint64_t)BH};
  cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)N * d * 2};
  cuuint32_t box[3] = {64, (cuuint32_t)box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
                   const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool aligned16(const void* p) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

fa_status check_shape(int B, int H, int N, int d, int dtype) {
  if (B < 1 || H < 1 || N < 1) return FA_ERR_INVALID_ARG;
  if (dtype != FA_FP16 && dtype != FA_BF16) return FA_ERR_UNSUPPORTED;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  const long long elems = (long long)B * H * N * d;
  if (elems >= (1LL << 31)) return FA_ERR_UNSUPPORTED;
  return FA_OK;
}

fa_status check_scale(float scale) {
  return (isfinite(scale) && scale > 0.f) ? FA_OK : FA_ERR_INVALID_ARG;
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

constexpr float kLog2e = 1.4426950408889634f;

}  // namespace

extern "C" {

const char* fa_status_string(int status) {
  switch (status) {
    case FA_OK: return "FA_OK";
    case FA_ERR_INVALID_ARG: return "FA_ERR_INVALID_ARG: null/misaligned pointer, bad size or bad scale";
    case FA_ERR_UNSUPPORTED: return "FA_ERR_UNSUPPORTED: head dim must be 64 or 128, dtype fp16/bf16, B*H*N*d < 2^31";
    case FA_ERR_CUDA: return "FA_ERR_CUDA: a CUDA launch or the stream failed";
    case FA_ERR_TIMEOUT: return "FA_ERR_TIMEOUT: a kernel gave up waiting on its pipeline";
    case FA_ERR_WORKSPACE: return "FA_ERR_WORKSPACE: workspace missing, misaligned or too small";
    case FA_ERR_SCRATCH_TOO_SMALL:
      return "FA_ERR_SCRATCH_TOO_SMALL: fa_backward_noalloc needs more than its fixed 32 MiB scratch; use fa_backward";
    default: return "unknown fa_status";
  }
}

}  // extern "C"

namespace {

// Dropout probability -> generator parameters: t = round(p * 65536), keep
// scale 65536 / (65536 - t).  False for p outside [0, 1) (NaN included) or
// p rounding to 1.
bool make_drop(float p, uint64_t seed, uint32_t offset, fa::DropParams* dp) {
  if (!(p >= 0.f && p < 1.f)) return false;
  const double t = floor((double)p * 65536.0 + 0.5);
  if (t >= 65536.0) return false;
  dp->t = (uint32_t)t;
  dp->keep_scale = (float)(65536.0 / (65536.0 - t));
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

fa_status forward_impl(const void* q, const void* k, const void* v, void* o, float* lse, const uint8_t* block_mask,
                       int mask_heads, int B, int H, int N, int d, int dtype, int causal, float scale,
                       void* stream, const fa::DropParams* drop = nullptr) {
  fa_status st = check_shape(B, H, N, d, dtype);
  if (st != FA_OK) return st;
  if ((st = check_scale(scale)) != FA_OK) return st;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
    return FA_ERR_INVALID_ARG;
  const bool bf16 = dtype == FA_BF16;
  fa::FwdArgs a;
  const int BH = B * H;
  if (!make_map(&a.tm_q, q, bf16, d, N, BH, 128) || !make_map(&a.tm_k, k, bf16, d, N, BH, 128) ||
      !make_map(&a.tm_v, v, bf16, d, N, BH, 128))
    return FA_ERR_CUDA;
  a.o = o;
  a.lse = lse;
  a.N = N;
  a.BH = BH;
  a.scale_log2 = scale * kLog2e;
  a.block_mask = block_mask;
  a.mask_heads = mask_heads;
  a.status = status_word();
  if (!a.status) return FA_ERR_CUDA;
  // p rounding to 0 drops nothing: the plain kernel computes exactly that.
  a.dropout = drop != nullptr && drop->t > 0;
  if (a.dropout) a.drop = *drop;
  const cudaError_t e = a.dropout ? fa::launch_forward_dropout(d, causal != 0, bf16, a, static_cast<cudaStream_t>(stream))
                                  : fa::launch_forward(d, causal != 0, bf16, a, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return FA_ERR_CUDA;
  return FA_OK;
}

}  // namespace

extern "C" {

fa_status fa_forward(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N,
                     int d, int dtype, int causal, float scale, void* stream) {
  return forward_impl(q, k, v, o, lse, nullptr, 1, B, H, N, d, dtype, causal, scale, stream);
}

fa_status fa_forward_blocksparse(const void* q, const void* k, const void* v, void* o, float* lse,
                                 const uint8_t* block_mask, int mask_heads, int B, int H, int N, int d, int dtype,
                                 int causal, float scale, void* stream) {
  const fa_status st = check_block_mask(block_mask, mask_heads, B, H);
  if (st != FA_OK) return st;
  return forward_impl(q, k, v, o, lse, block_mask, mask_heads, B, H, N, d, dtype, causal, scale, stream);
}

size_t fa_backward_workspace_size(int B, int H, int N, int d) {
  if (check_shape(B, H, N, d, FA_BF16) != FA_OK) return 0;
  const size_t rows = (size_t)B * H * N;
  return align256(rows * sizeof(float)) + align256(rows * d * sizeof(float));
}

fa_status fa_backward_preprocess(const void* o, const void* dO, float* delta, float* dq_accum, int B, int H,
                                 int N, int d, int dtype, void* stream) {
  fa_status st = check_shape(B, H, N, d, dtype);
  if (st != FA_OK) return st;
  if (!aligned16(o) || !aligned16(dO) || !aligned16(delta) || !aligned16(dq_accum)) return FA_ERR_INVALID_ARG;
  const long long rows = (long long)B * H * N;
  if (fa::launch_backward_preprocess(d, dtype == FA_BF16, o, dO, delta, dq_accum, rows,
                                     static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return FA_ERR_CUDA;
  return FA_OK;
}

}  // extern "C"

namespace {

fa_status dkdv_impl(const void* q, const void* k, const void* v, const void* dO, const float* lse, const float* delta,
                    float* dq_accum, void* dk, void* dv, const uint8_t* block_mask, int mask_heads, int B, int H,
                    int N, int d, int dtype, int causal, float scale, void* stream,
                    const fa::DropParams* drop = nullptr) {
  fa_status st = check_shape(B, H, N, d, dtype);
  if (st != FA_OK) return st;
  if ((st = check_scale(scale)) != FA_OK) return st;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(dO) || !aligned16(lse) ||
      !aligned16(delta) || !aligned16(dq_accum) || !aligned16(dk) || !aligned16(dv))
    return FA_ERR_INVALID_ARG;
  const bool bf16 = dtype == FA_BF16;
  const int BH = B * H;
  const int bq = fa::backward_q_tile(d);
  fa::BwdArgs a;
  if (!make_map(&a.tm_q, q, bf16, d, N, BH, bq) || !make_map(&a.tm_do, dO, bf16, d, N, BH, bq) ||
      !make_map(&a.tm_k, k, bf16, d, N, BH, 128) || !make_map(&a.tm_v, v, bf16, d, N, BH, 128))
    return FA_ERR_CUDA;
  a.dk = dk;
  a.dv = dv;
  a.lse = lse;
  a.delta = delta;
  a.dq_accum = dq_accum;
  a.N = N;
  a.BH = BH;
  a.scale = scale;
  a.scale_log2 = scale * kLog2e;
  a.block_mask = block_mask;
  a.mask_heads = mask_heads;
  a.status = status_word();
  if (!a.status) return FA_ERR_CUDA;
  a.dropout = drop != nullptr && drop->t > 0;
  if (a.dropout) a.drop = *drop;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  const cudaError_t e = a.dropout ? fa::launch_backward_dkdv_dropout(d, causal != 0, bf16, a, s)
                                  : fa::launch_backward_dkdv(d, causal != 0, bf16, a, s);
  if (e != cudaSuccess) return FA_ERR_CUDA;
  return FA_OK;
}

}  // namespace

extern "C" {

fa_status fa_backward_dkdv(const void* q, const void* k, const void* v, const void* dO, const float* lse,
                           const float* delta, float* dq_accum, void* dk, void* dv, int B, int H, int N, int d,
                           int dtype, int causal, float scale, void* stream) {
  return dkdv_impl(q, k, v, dO, lse, delta, dq_accum, dk, dv, nullptr, 1, B, H, N, d, dtype, causal, scale, stream);
}

fa_status fa_backward_dkdv_blocksparse(const void* q, const void* k, const void* v, const void* dO, const float* lse,
                                       const float* delta, float* dq_accum, void* dk, void* dv,
                                       const uint8_t* block_mask, int mask_heads, int B, int H, int N, int d,
                                       int dtype, int causal, float scale, void* stream) {
  const fa_status st = check_block_mask(block_mask, mask_heads, B, H);
  if (st != FA_OK) return st;
  return dkdv_impl(q, k, v, dO, lse, delta, dq_accum, dk, dv, block_mask, mask_heads, B, H, N, d, dtype, causal,
                   scale, stream);
}

fa_status fa_backward_dq_convert(const float* dq_accum, void* dq, int B, int H, int N, int d, int dtype,
                                 float scale, void* stream) {
  fa_status st = check_shape(B, H, N, d, dtype);
  if (st != FA_OK) return st;
  if ((st = check_scale(scale)) != FA_OK) return st;
  if (!aligned16(dq_accum) || !aligned16(dq)) return FA_ERR_INVALID_ARG;
  const long long rows = (long long)B * H * N;
  if (fa::launch_backward_dq_convert(d, dtype == FA_BF16, dq_accum, dq, rows, scale,
                                     static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return FA_ERR_CUDA;
  return FA_OK;
}

}  // extern "C"

namespace {

fa_status backward_impl(const void* q, const void* k, const void* v, const void* o, const void* dO, const float* lse,
                        void* dq, void* dk, void* dv, const uint8_t* block_mask, int mask_heads, int B, int H, int N,
                        int d, int dtype, int causal, float scale, void* workspace, size_t workspace_bytes,
                        void* stream, const fa::DropParams* drop = nullptr) {
  fa_status st = check_shape(B, H, N, d, dtype);
  if (st != FA_OK) return st;
  if ((st = check_scale(scale)) != FA_OK) return st;
  const size_t need = fa_backward_workspace_size(B, H, N, d);
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) || workspace_bytes < need)
    return FA_ERR_WORKSPACE;
  const size_t rows = (size_t)B * H * N;
  float* delta = static_cast<float*>(workspace);
  float* dq_accum = reinterpret_cast<float*>(static_cast<char*>(workspace) + align256(rows * sizeof(float)));
  if ((st = fa_backward_preprocess(o, dO, delta, dq_accum, B, H, N, d, dtype, stream)) != FA_OK) return st;
  if ((st = dkdv_impl(q, k, v, dO, lse, delta, dq_accum, dk, dv, block_mask, mask_heads, B, H, N, d, dtype, causal,
                      scale, stream, drop)) != FA_OK)
    return st;
  return fa_backward_dq_convert(dq_accum, dq, B, H, N, d, dtype, scale, stream);
}

}  // namespace

extern "C" {

fa_status fa_backward(const void* q, const void* k, const void* v, const void* o, const void* dO,
                      const float* lse, void* dq, void* dk, void* dv, int B, int H, int N, int d, int dtype,
                      int causal, float scale, void* workspace, size_t workspace_bytes, void* stream) {
  return backward_impl(q, k, v, o, dO, lse, dq, dk, dv, nullptr, 1, B, H, N, d, dtype, causal, scale, workspace,
                       workspace_bytes, stream);
}

fa_status fa_backward_blocksparse(const void* q, const void* k, const void* v, const void* o, const void* dO,
                                  const float* lse, void* dq, void* dk, void* dv, const uint8_t* block_mask,
                                  int mask_heads, int B, int H, int N, int d, int dtype, int causal, float scale,
                                  void* workspace, size_t workspace_bytes, void* stream) {
  const fa_status st = check_block_mask(block_mask, mask_heads, B, H);
  if (st != FA_OK) return st;
  return backward_impl(q, k, v, o, dO, lse, dq, dk, dv, block_mask, mask_heads, B, H, N, d, dtype, causal, scale,
                       workspace, workspace_bytes, stream);
}

namespace {
fa_status decode_plan(int B, int H, int Nq, int Nk, int d, int num_splits, int* splits, int* chunk,
                      size_t* bytes) {
  if (B < 1 || H < 1 || Nq < 1 || Nk < 1) return FA_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
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

size_t fa_decode_workspace_size(int B, int H, int Nq, int Nk, int d, int num_splits) {
  int s, c;
  size_t bytes = 0;
  return decode_plan(B, H, Nq, Nk, d, num_splits, &s, &c, &bytes) == FA_OK ? bytes : 0;
}

fa_status fa_forward_decode(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                            int Nq, int Nk, int d, int dtype, int causal, float scale, int num_splits,
                            void* workspace, size_t workspace_bytes, void* stream) {
  int splits, chunk;
  size_t need;
  fa_status st = decode_plan(B, H, Nq, Nk, d, num_splits, &splits, &chunk, &need);
  if (st != FA_OK) return st;
  if (dtype != FA_FP16 && dtype != FA_BF16) return FA_ERR_UNSUPPORTED;
  if ((st = check_scale(scale)) != FA_OK) return st;
  if (causal && Nq > Nk) return FA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
    return FA_ERR_INVALID_ARG;
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) || workspace_bytes < need)
    return FA_ERR_WORKSPACE;
  fa::DecodeArgs a;
  a.q = q;
  a.k = k;
  a.v = v;
  a.o = o;
  a.lse = lse;
  a.BH = B * H;
  a.Nq = Nq;
  a.Nk = Nk;
  a.num_splits = splits;
  a.chunk = chunk;
  a.causal = causal != 0;
  a.scale_log2 = scale * kLog2e;
  const size_t rows = (size_t)splits * a.BH * Nq;
  a.o_part = static_cast<float*>(workspace);
  a.lse_part = reinterpret_cast<float*>(static_cast<char*>(workspace) + align256(rows * d * sizeof(float)));
  if (fa::launch_decode(d, dtype == FA_BF16, a, static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return FA_ERR_CUDA;
  return FA_OK;
}

fa_status fa_forward_dropout(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N,
                             int d, int dtype, int causal, float scale, float p_drop, uint64_t seed,
                             uint32_t offset, void* stream) {
  fa::DropParams dp;
  if (!make_drop(p_drop, seed, offset, &dp)) return FA_ERR_INVALID_ARG;
  return forward_impl(q, k, v, o, lse, nullptr, 1, B, H, N, d, dtype, causal, scale, stream, &dp);
}

fa_status fa_backward_dropout(const void* q, const void* k, const void* v, const void* o, const void* dO,
                              const float* lse, void* dq, void* dk, void* dv, int B, int H, int N, int d, int dtype,
                              int causal, float scale, float p_drop, uint64_t seed, uint32_t offset, void* workspace,
                              size_t workspace_bytes, void* stream) {
  fa::DropParams dp;
  if (!make_drop(p_drop, seed, offset, &dp)) return FA_ERR_INVALID_ARG;
  return backward_impl(q, k, v, o, dO, lse, dq, dk, dv, nullptr, 1, B, H, N, d, dtype, causal, scale, workspace,
                       workspace_bytes, stream, &dp);
}

fa_status fa_backward_dkdv_dropout(const void* q, const void* k, const void* v, const void* dO, const float* lse,
                                   const float* delta, float* dq_accum, void* dk, void* dv, int B, int H, int N,
                                   int d, int dtype, int causal, float scale, float p_drop, uint64_t seed,
                                   uint32_t offset, void* stream) {
  fa::DropParams dp;
  if (!make_drop(p_drop, seed, offset, &dp)) return FA_ERR_INVALID_ARG;
  return dkdv_impl(q, k, v, dO, lse, delta, dq_accum, dk, dv, nullptr, 1, B, H, N, d, dtype, causal, scale, stream,
                   &dp);
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

fa_status fa_device_status(void* stream) {
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return FA_ERR_CUDA;
  unsigned int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_fa_status, sizeof(v)) != cudaSuccess) return FA_ERR_CUDA;
  if (v != 0) {
    const unsigned int zero = 0;
    if (cudaMemcpyToSymbol(g_fa_status, &zero, sizeof(zero)) != cudaSuccess) return FA_ERR_CUDA;
    if (v & fa::kStatusTimeout) return FA_ERR_TIMEOUT;
  }
  return FA_OK;
}

}  // extern "C"
