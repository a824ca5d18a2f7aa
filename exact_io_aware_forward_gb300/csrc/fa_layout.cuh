// Device view of one (sequence, head) problem of a SeqLayout (fa_internal.h):
// its lengths, the TMA coordinates of its rows and the flat row index of a
// row in the [rows, dh] view of O, dQ, dK, dV (and of LSE / D).
#pragma once

#include "fa_internal.h"

namespace fa {

struct SeqView {
  int nq, nk;                 // query and key rows of this problem
  int qrow0, krow0;           // first packed row (varlen), 0 (dense)
  int z;                      // third TMA coordinate (dense: b*H + h) or head (varlen)
  long long qflat0, kflat0;   // flat row of row 0
  int rstride;                // flat rows between consecutive rows: 1 (dense), H (varlen)
  bool varlen;
  bool ok;                    // false: the offsets of this sequence are out of range

  // TMA (y, z) coordinates of query / key row r.  Dense maps are
  // (d, N, B*H); varlen maps are (d, H, T) so that their strides increase.
  __device__ __forceinline__ int2 qcoord(int r) const {
    return varlen ? make_int2(z, qrow0 + r) : make_int2(r, z);
  }
  __device__ __forceinline__ int2 kcoord(int r) const {
    return varlen ? make_int2(z, krow0 + r) : make_int2(r, z);
  }
  __device__ __forceinline__ long long qflat(int r) const { return qflat0 + (long long)r * rstride; }
  __device__ __forceinline__ long long kflat(int r) const { return kflat0 + (long long)r * rstride; }
};

// VARLEN is the kernel's compile-time choice (the dense instances never read
// offsets and see rstride = 1 as a constant).
template <bool VARLEN>
__device__ __forceinline__ SeqView seq_view(const SeqLayout& L, int bh) {
  SeqView v;
  if (VARLEN) {
    const int b = bh / L.H, h = bh % L.H;
    v.varlen = true;
    v.qrow0 = L.cu_q[b];
    v.nq = L.cu_q[b + 1] - v.qrow0;
    v.krow0 = L.cu_k[b];
    v.nk = L.cu_k[b + 1] - v.krow0;
    v.ok = v.qrow0 >= 0 && v.krow0 >= 0 && v.nq >= 0 && v.nk >= 0 && v.nq <= L.Nq && v.nk <= L.Nk &&
           v.qrow0 + v.nq <= L.Tq && v.krow0 + v.nk <= L.Tk;
    if (!v.ok) v.nq = v.nk = 0;  // skipped; the caller reports it
    v.z = h;
    v.qflat0 = (long long)v.qrow0 * L.H + h;
    v.kflat0 = (long long)v.krow0 * L.H + h;
    v.rstride = L.H;
  } else {
    v.varlen = false;
    v.ok = true;
    v.qrow0 = v.krow0 = 0;
    v.nq = L.Nq;
    v.nk = L.Nk;
    v.z = bh;
    v.qflat0 = (long long)bh * L.Nq;
    v.kflat0 = (long long)bh * L.Nk;
    v.rstride = 1;
  }
  return v;
}

// Number of 128-key tiles [0, n) that contain a key visible to some query row
// <= last_row under the bottom-right causal mask (key <= row + off,
// off = nk - nq), out of n_kv tiles.
__device__ __forceinline__ int causal_key_tiles(int last_row, int off, int n_kv, int tile) {
  const int last_key = last_row + off;
  if (last_key < 0) return 0;
  const int n = last_key / tile + 1;
  return n < n_kv ? n : n_kv;
}

}  // namespace fa
