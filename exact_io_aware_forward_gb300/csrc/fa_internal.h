// Launch interfaces between the C-ABI translation unit and the kernel
// translation units.  Not part of the public interface.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace fa {

// Status bits latched by kernels in the device status word.
constexpr unsigned int kStatusTimeout = 1u;
constexpr unsigned int kStatusBadSeqlens = 2u;  // a cu_seqlens range outside the packed tensors or maxima

// The device status block: word 0 holds the kStatus* bits; words 2-3 and 4-5
// are two 64-bit counters of the 64 x 64 (query x key) score blocks that the
// forward and the backward kernels computed.  Kernels get a pointer to word 0.
constexpr int kStatusWords = 6;
constexpr int kCountForward = 0;
constexpr int kCountBackward = 1;

#ifdef __CUDACC__
// Adds n score blocks to counter `which` (kCountForward / kCountBackward).
__device__ __forceinline__ void count_score_blocks(unsigned int* status, int which, unsigned long long n) {
  atomicAdd(reinterpret_cast<unsigned long long*>(status + 2) + which, n);
}
#endif

// Where the rows of each (sequence, head) problem live.
//   dense  (cu_q == nullptr): q/o/dq [B, H, Nq, dh], k/v/dk/dv [B, H, Nk, dh]
//          head-major, every sequence of the same length; lse/delta [B, H, Nq].
//   varlen (cu_q != nullptr): packed token-major q/o/dq [Tq, H, dh] and
//          k/v/dk/dv [Tk, H, dh]; sequence b owns query rows cu_q[b] ..
//          cu_q[b+1]-1 and key rows cu_k[b] .. cu_k[b+1]-1; lse/delta [Tq, H].
//          Nq / Nk are then the largest sequence lengths (grid sizing only).
// dh is the head dimension of the tensors; the kernels compute with width
// D >= dh (dh = 96 runs the D = 128 kernels with the features 96-127 read
// as zero by TMA and never stored).
struct SeqLayout {
  const int* cu_q = nullptr;
  const int* cu_k = nullptr;
  int H = 1;
  int Nq = 0, Nk = 0;
  int Tq = 0, Tk = 0;  // varlen: packed rows of q and k (bounds for the offsets)
  int dh = 0;
};

// Dropout parameters (see fa_philox.cuh): entries whose 8-bit draw is below
// t are dropped; kept ones are scaled by keep_scale = 256 / (256 - t).
struct DropParams {
  uint32_t t = 0;
  float keep_scale = 1.f;
  uint32_t k0 = 0, k1 = 0;  // generator key: seed low and high words
  uint32_t offset = 0;      // counter word 3
};

struct FwdArgs {
  CUtensorMap tm_q, tm_k, tm_v;        // 3-D maps, box 64 columns x 128 rows (see make_map)
  CUtensorMap tm_o;                    // O, box 64 columns x 128 rows (TMA-stored epilogues)
  void* o;                             // layout `lay`
  float* lse;
  SeqLayout lay;
  int BH;                              // B * H
  float scale_log2;                    // scale * log2(e)
  const uint8_t* block_mask = nullptr; // [mask_heads, T, T] block mask, T = ceil(N/128); null = dense
  int mask_heads = 1;                  // 1 (shared by all heads) or B*H
  bool dropout = false;                // apply `drop` (dense attention only)
  DropParams drop;
  unsigned int* status;                // device status word
};
cudaError_t launch_forward(int d, bool causal, bool bf16, const FwdArgs& a, cudaStream_t stream);
// Dense layouts without block mask or dropout: the persistent kernel (a CTA
// takes further work items from CTAs of its grid that have not started).
cudaError_t launch_forward_persistent(int d, bool causal, bool bf16, const FwdArgs& a, cudaStream_t stream);
cudaError_t launch_forward_dropout(int d, bool causal, bool bf16, const FwdArgs& a, cudaStream_t stream);
// Packed variable-length instances (a.lay.cu_q != nullptr), with or without dropout.
cudaError_t launch_forward_varlen(int d, bool causal, bool bf16, const FwdArgs& a, cudaStream_t stream);
// Head dimension 256 (dense or packed, with or without dropout; no block mask).
cudaError_t launch_forward256(bool causal, bool bf16, const FwdArgs& a, cudaStream_t stream);

struct BwdArgs {
  CUtensorMap tm_q, tm_do;         // box 64 columns x BQ rows
  CUtensorMap tm_k, tm_v;          // box 64 columns x 128 rows
  CUtensorMap tm_dk, tm_dv;        // box 64 columns x 128 rows (dense layouts: epilogue stores)
  void* dk;                        // layout `lay` (key side)
  void* dv;
  const float* lse;                // one float per query row
  const float* delta;
  float* dq_accum;                 // float32, query side, dh columns
  SeqLayout lay;
  int BH;
  float scale;
  float scale_log2;
  const uint8_t* block_mask = nullptr;  // as FwdArgs
  int mask_heads = 1;
  bool dropout = false;                 // as FwdArgs
  DropParams drop;
  unsigned int* status;
};
// The status fa_backward returns for these arguments before it looks at its
// workspace (FA_OK when shape, dtype, scale and every pointer are valid).
int backward_arguments_status(const void* q, const void* k, const void* v, const void* o, const void* dO,
                              const float* lse, const void* dq, const void* dk, const void* dv, int B, int H, int N,
                              int d, int dtype, float scale);
int backward_q_tile(int d);  // query rows per inner iteration of the dK/dV kernel
cudaError_t launch_backward_dkdv(int d, bool causal, bool bf16, const BwdArgs& a, cudaStream_t stream);
cudaError_t launch_backward_dkdv_dropout(int d, bool causal, bool bf16, const BwdArgs& a, cudaStream_t stream);
cudaError_t launch_backward_dkdv_varlen(int d, bool causal, bool bf16, const BwdArgs& a, cudaStream_t stream);
// keep[bh][i][j] = 1 if entry (bh, i, j) is kept, else 0 ([BH, Nq, Nk] bytes).
cudaError_t launch_dropout_keep_mask(uint8_t* keep, int BH, int Nq, int Nk, const DropParams& drop,
                                     cudaStream_t stream);
// The backward pass with dQ computed by a kernel of its own (dense layouts
// with a block mask, with dropout or with neither; packed variable-length
// batches without dropout): a dK / dV kernel and a dQ kernel that both
// recompute P and dP on chip.
struct SplitArgs {
  CUtensorMap tm_q, tm_do;         // box 64 columns x 128 rows
  CUtensorMap tm_k, tm_v;          // box 64 columns x 128 rows
  CUtensorMap tm_dk, tm_dv;        // box 64 columns x 128 rows (epilogue stores)
  void* dq;                        // layout `lay` (query side), 16-bit
  void* dk;                        // layout `lay` (key side): packed layouts store rows one by one
  void* dv;
  const float* lse;
  const float* delta;
  SeqLayout lay;
  int BH, dh;
  float scale, scale_log2;
  const uint8_t* block_mask = nullptr;  // as FwdArgs (128 x 128 blocks); null = dense
  int mask_heads = 1;
  bool dropout = false;                 // apply `drop` (dense layouts only)
  DropParams drop;
  unsigned int* status;
};
cudaError_t launch_backward_dkdv_split(int d, bool causal, bool bf16, const SplitArgs& a, cudaStream_t stream);
cudaError_t launch_backward_dq(int d, bool causal, bool bf16, const SplitArgs& a, cudaStream_t stream);
cudaError_t launch_backward_preprocess(int d, bool bf16, const void* o, const void* dO, float* delta,
                                       float* dq_accum, long long rows, cudaStream_t stream);
cudaError_t launch_backward_dq_convert(int d, bool bf16, const float* dq_accum, void* dq, long long rows,
                                       float scale, cudaStream_t stream);
// One thread waits, with the kernels' bounded wait, on an mbarrier that no
// one arrives at; the wait gives up and latches kStatusTimeout in *status.
cudaError_t launch_selftest_wait_timeout(unsigned int* status, cudaStream_t stream);

struct DecodeArgs {
  void* o;             // [B*H, Nq, d]
  float* lse;          // [B*H, Nq]
  float* o_part;       // [num_splits, B*H, Nq, d] float32
  float* lse_part;     // [num_splits, B*H, Nq] float32, log2 units
  int BH, Nq, Nk;
  int num_splits;
  int chunk;           // keys per split (multiple of 256)
  bool causal;
  float scale_log2;
  CUtensorMap tm_q, tm_k, tm_v;  // 3-D maps over q, k, v, box 64 columns x 128 rows
  unsigned int* status = nullptr;
};
// Decoding runs on the tensor cores (fa_decode_tc.cu) at every head dimension:
// streaming K and V it reached 85-91% of the HBM bandwidth from 1 to 64 queries
// per head at d = 128 and d = 256, where a CUDA-core kernel (dot products of
// up to 16 queries per key row on the FMA pipe) reached 78-80% at one query,
// 18% at 16 and 5% at 64.
int decode_default_splits(int BH, int Nq, int Nk);
int decode_chunk(int Nk, int num_splits);
cudaError_t launch_decode_tc(int d, bool bf16, const DecodeArgs& a, cudaStream_t stream);
cudaError_t launch_decode_combine(int d, bool bf16, const DecodeArgs& a, cudaStream_t stream);

}  // namespace fa
