// The multi-column block-quantized GEMV engine shared by the dense GEMV and
// the grouped MoE decode kernels.
//
// What it computes (#242 What it does; #1424 What changed): for a weight row
// r and activation column c,
//   y[c][r] = sum_b fp32(dw[r,b]) * dx[c,b] * I[c,r,b],
//   I[c,r,b] = sum_{i<32} qw[r,32b+i] * qx[c,32b+i]   (int32, dp4a chains)
// Each weight block is read from shared memory and decoded once per pass and
// applied to every column of the pass (the "load once, apply per column"
// split of #242).
//
// GB300 layout (not the pages' warp-per-row kernels):
//  * a single producer thread streams contiguous row ranges of the weight
//    planes into a ring of shared-memory stages with cp.async.bulk (16-byte
//    aligned bulk copies completing on mbarriers), so each SM keeps tens of
//    KB of HBM reads in flight from the first cycle;
//  * the K axis is cut into slices of 16 blocks; a consumer warp owns one
//    slice and its 16 lanes x 2 halves hold one 32-value block each, with the
//    activations of that block for all columns in registers (loaded once per
//    column set), so activations cost no shared-memory traffic per row;
//  * a stage of 8 rows is shared by all consumer warps (every slice, every
//    row), so the last stage to arrive is finished quickly;
//  * per-lane partial sums are reduced over the 16 lanes with a recursive
//    halving exchange (xor 8, 4, 2, 1) whose summation tree does not depend
//    on the number of columns, then over the slices in slice order, so a
//    column's result is bitwise the same for any column count (#242 / #1424:
//    every column of a multi-column call equals a one-column call).
#pragma once

#include <cuda_fp16.h>

#include "common.cuh"

namespace moex {

constexpr int SR = 8;        // rows per pipeline stage
constexpr int SLICE = 16;    // blocks per K slice (one per lane of a half warp)

__host__ __device__ inline int64_t qs_row_bytes(int fmt, int64_t K) { return fmt == MOEX_Q8_0 ? K : K / 2; }
__host__ __device__ inline int64_t sc_row_bytes(int64_t K) { return ((K / QK) * 2 + 15) / 16 * 16; }

template <int FMT>
struct FmtTraits;
template <>
struct FmtTraits<MOEX_Q8_0> {
  static constexpr int QBYTES = 32;  // quant bytes per block
};
template <>
struct FmtTraits<MOEX_IQ4_NL> {
  static constexpr int QBYTES = 16;
};

// ----------------------------------------------------------------- activations

// Per-lane activation registers for one block b and C columns.
//  Q8_0 lanes read their weight block as two 16-byte halves in the order
//  h0 = (li >> 2) & 1, then 1 - h0 (this spreads the 8 lanes of a shared
//  memory phase over all 32 banks); the activation words are held in the
//  same order.
//  IQ4_NL weights decode to the byte order x[j], x[j+16], x[j+1], x[j+17]
//  (low and high nibble of consecutive index bytes); the activation words
//  are held permuted to match:
//    A[2i]   = x[4i],   x[4i+16], x[4i+1], x[4i+17]
//    A[2i+1] = x[4i+2], x[4i+18], x[4i+3], x[4i+19]
template <int FMT, int C>
struct ActRegs {
  uint32_t a[C][8];
  float d[C];
};

// Loads activations of block b (natural order: column c's quants at
// xcol[c], its scales at dcol[c]; dcol == nullptr gives unit scales) into
// registers.  Invalid blocks get zeros.
template <int FMT, int C>
__device__ __forceinline__ void load_act(ActRegs<FMT, C>& r, const int8_t* const* xcol, const float* const* dcol,
                                         int b, bool valid, int li) {
#pragma unroll
  for (int c = 0; c < C; ++c) {
    if (!valid) {
#pragma unroll
      for (int i = 0; i < 8; ++i) r.a[c][i] = 0u;
      r.d[c] = 0.f;
      continue;
    }
    const int8_t* src = xcol[c] + b * QK;
    uint4 lo = *reinterpret_cast<const uint4*>(src);
    uint4 hi = *reinterpret_cast<const uint4*>(src + 16);
    if constexpr (FMT == MOEX_Q8_0) {
      const bool swap = (li >> 2) & 1;
      const uint4 f = swap ? hi : lo;
      const uint4 s = swap ? lo : hi;
      r.a[c][0] = f.x; r.a[c][1] = f.y; r.a[c][2] = f.z; r.a[c][3] = f.w;
      r.a[c][4] = s.x; r.a[c][5] = s.y; r.a[c][6] = s.z; r.a[c][7] = s.w;
    } else {
      const uint32_t X[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        r.a[c][2 * i] = prmt(X[i], X[i + 4], 0x5140);
        r.a[c][2 * i + 1] = prmt(X[i], X[i + 4], 0x7362);
      }
    }
    r.d[c] = dcol ? dcol[c][b] : 1.f;
  }
}

// ----------------------------------------------------------------- one row

// Integer dots of one weight block (row pointer at the block) with C columns,
// then p[c] = I * (dw * dx[c]) in FP32.
template <int FMT, int C>
__device__ __forceinline__ void block_row_dots(const uint8_t* wq, float dw, const ActRegs<FMT, C>& act, int li,
                                               float* p, int* I_out = nullptr) {
  uint32_t wv[8];
  if constexpr (FMT == MOEX_Q8_0) {
    const int h0 = (li >> 2) & 1;
    const uint4 f = *reinterpret_cast<const uint4*>(wq + 16 * h0);
    const uint4 s = *reinterpret_cast<const uint4*>(wq + 16 * (1 - h0));
    wv[0] = f.x; wv[1] = f.y; wv[2] = f.z; wv[3] = f.w;
    wv[4] = s.x; wv[5] = s.y; wv[6] = s.z; wv[7] = s.w;
  } else {
    const uint4 n = *reinterpret_cast<const uint4*>(wq);
    const uint32_t W[4] = {n.x, n.y, n.z, n.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t fl = W[i] ^ 0x88888888u;
      wv[2 * i] = iq4nl_lookup4(W[i], fl);
      wv[2 * i + 1] = iq4nl_lookup4(W[i] >> 16, fl >> 16);
    }
  }
#pragma unroll
  for (int c = 0; c < C; ++c) {
    int I = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) I = dp4a(wv[i], act.a[c][i], I);
    if (I_out) I_out[c] = I;
    p[c] = __fmul_rn(__int2float_rn(I), __fmul_rn(dw, act.d[c]));
  }
}

// ----------------------------------------------------------------- reduction

// Recursive-halving sum of N values per lane over the 16 lanes of each half
// warp (xor offsets 8, 4, 2, 1).  Value v ends up summed with the same tree
// (pairs by lane bit 3, then 2, 1, 0) for every N.  Afterwards, for N >= 16,
// lane li holds values li*(N/16) + i in v[i]; for N < 16 it holds value
// li / (16/N) in v[0].
template <int N, int O>
__device__ __forceinline__ void halving_reduce(float* v, int lane) {
  if constexpr (O > 0) {
    if constexpr (N > 1) {
      const bool upper = (lane & O) != 0;
#pragma unroll
      for (int i = 0; i < N / 2; ++i) {
        const float send = upper ? v[i] : v[i + N / 2];
        const float keep = upper ? v[i + N / 2] : v[i];
        v[i] = keep + __shfl_xor_sync(0xffffffffu, send, O);
      }
      halving_reduce<N / 2, O / 2>(v, lane);
    } else {
      v[0] = v[0] + __shfl_xor_sync(0xffffffffu, v[0], O);
      halving_reduce<1, O / 2>(v, lane);
    }
  }
}

__host__ __device__ constexpr int pow2_ceil(int v) { return v <= 1 ? 1 : 2 * pow2_ceil((v + 1) / 2); }

// ----------------------------------------------------------------- consumer layout

// Consumer warp w owns slice ks = w / WPS; its half `hf` (lane >> 4) and
// index jw = w % WPS give the stage rows jw*2 + hf + 2*WPS*i, i < RPH, with
// RPH = SR / (2*WPS).
struct ConsumerPos {
  int ks, jw, hf, li, lane;
};

// Computes one stage for one consumer warp and writes its per-slice partial
// sums red[row][ks][c] (row < nrows).  wq_stage / sc_stage are the stage's
// quant rows (stride qrow bytes) and FP16 scale rows (stride scrow bytes).
template <int FMT, int C, int WPS>
__device__ __forceinline__ void stage_partials(const uint8_t* wq_stage, const uint8_t* sc_stage, int qrow, int scrow,
                                               int nrows, int NB, int NS, const ConsumerPos& pos,
                                               const ActRegs<FMT, C>& act, float* red) {
  constexpr int RPH = SR / (2 * WPS);
  constexpr int V = RPH * C;
  constexpr int N = pow2_ceil(V);
  float v[N];
#pragma unroll
  for (int i = 0; i < N; ++i) v[i] = 0.f;
  const int b = pos.ks * SLICE + pos.li;
  const bool bvalid = b < NB;
#pragma unroll
  for (int rr = 0; rr < RPH; ++rr) {
    const int row = pos.jw * 2 + pos.hf + 2 * WPS * rr;
    if (bvalid && row < nrows) {
      const uint8_t* wq = wq_stage + row * qrow + b * FmtTraits<FMT>::QBYTES;
      const float dw = __half2float(reinterpret_cast<const __half*>(sc_stage + row * scrow)[b]);
      block_row_dots<FMT, C>(wq, dw, act, pos.li, &v[rr * C]);
    }
  }
  halving_reduce<N, 8>(v, pos.lane);
  // scatter to red[row][ks][c]
  const int li = pos.li;
  if constexpr (N >= 16) {
#pragma unroll
    for (int i = 0; i < N / 16; ++i) {
      const int idx = li * (N / 16) + i;
      if (idx < V) {
        const int rr = idx / C, c = idx % C;
        const int row = pos.jw * 2 + pos.hf + 2 * WPS * rr;
        if (row < nrows) red[(row * NS + pos.ks) * C + c] = v[i];
      }
    }
  } else {
    constexpr int REP = 16 / N;
    if (li % REP == 0) {
      const int idx = li / REP;
      if (idx < V) {
        const int rr = idx / C, c = idx % C;
        const int row = pos.jw * 2 + pos.hf + 2 * WPS * rr;
        if (row < nrows) red[(row * NS + pos.ks) * C + c] = v[0];
      }
    }
  }
}

// Final sum over slices (in slice order) of red[row][ks][c] for one stage,
// run by one warp.  Calls out(row, c, value) for row < nrows, c < C.
template <int C, typename Out>
__device__ __forceinline__ void stage_final(const float* red, int nrows, int NS, int lane, Out&& out) {
  for (int idx = lane; idx < nrows * C; idx += 32) {
    const int row = idx / C, c = idx % C;
    float s = red[(row * NS + 0) * C + c];
    for (int ks = 1; ks < NS; ++ks) s = s + red[(row * NS + ks) * C + c];
    out(row, c, s);
  }
}

// Marks one consumer warp done with a stage; returns true for the last warp
// (which then owns the final sum).  Shared-memory counter per slot.
__device__ __forceinline__ bool stage_arrive_last(int* cnt, int nwarps, int lane) {
  int old = 0;
  __syncwarp();
  if (lane == 0) {
    __threadfence_block();
    old = atomicAdd(cnt, 1);
  }
  old = __shfl_sync(0xffffffffu, old, 0);
  const bool last = old == nwarps - 1;
  if (last) __threadfence_block();
  return last;
}

// Consumer warp count for a K with NB blocks, and warps per slice.
__host__ __device__ inline int num_slices(int NB) { return (NB + SLICE - 1) / SLICE; }
__host__ __device__ inline int warps_per_slice(int NS) { return NS <= 3 ? 4 : (NS <= 7 ? 2 : 1); }

}  // namespace moex
