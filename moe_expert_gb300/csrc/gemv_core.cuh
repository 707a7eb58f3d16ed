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
//  * the K axis is cut into slices of 16 blocks; a warp owns one slice and
//    its 16 lanes x 2 halves hold one 32-value block each, with the
//    activations of that block for all columns in registers (loaded once per
//    column set), so activations cost no shared-memory traffic per row;
//  * weights arrive in stages of 8 consecutive rows: either through a
//    shared-memory ring that one producer thread fills with two bulk (TMA)
//    copies a stage (the 8 rows' quants, then their scales), or, in the
//    register-staged GEMV, as each lane's own 16-byte loads of its block of
//    each row;
//  * a stage of 8 rows is shared by all warps (every slice, every row), so
//    the last stage to arrive is finished quickly;
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
//  Q8_0: the 8 words in natural order.
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
// xcol[c], its d scales at dcol[c][b * dstride]; dcol == nullptr gives unit
// scales) into registers.  Invalid blocks get zeros.  The pointers may be
// shared or global memory.  With `swap` (Q8_0 only) the two 16-byte halves
// of the block are held in swapped order, to match a weight block read with
// the same swap (the integer dot is the same sum in another order).
template <int FMT, int C>
__device__ __forceinline__ void load_act(ActRegs<FMT, C>& r, const int8_t* const* xcol, const float* const* dcol,
                                         int b, bool valid, int li, int dstride = 1, bool swap = false) {
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
      if (swap) {
        const uint4 t = lo;
        lo = hi;
        hi = t;
      }
      r.a[c][0] = lo.x; r.a[c][1] = lo.y; r.a[c][2] = lo.z; r.a[c][3] = lo.w;
      r.a[c][4] = hi.x; r.a[c][5] = hi.y; r.a[c][6] = hi.z; r.a[c][7] = hi.w;
    } else {
      const uint32_t X[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        r.a[c][2 * i] = prmt(X[i], X[i + 4], 0x5140);
        r.a[c][2 * i + 1] = prmt(X[i], X[i + 4], 0x7362);
      }
    }
    r.d[c] = dcol ? dcol[c][b * dstride] : 1.f;
  }
}

// ----------------------------------------------------------------- one row

// Integer dots of one weight block with C columns, then
// p[c] = I * (dw * dx[c]) in FP32.  The block's quant bytes are given as
// 16-byte chunks q0 (and q1 for Q8_0).
// SPLIT (IQ4_NL, C <= 2): two table lookups and two dp4a's per four weights
// (split codebook) instead of rebuilding the values: fewer instructions, but
// twice the dp4a's.
template <int FMT, int C, bool SPLIT = false>
__device__ __forceinline__ void block_dots_from(uint4 q0, uint4 q1, float dw, const ActRegs<FMT, C>& act, float* p,
                                                int* I_out = nullptr) {
  if constexpr (FMT != MOEX_Q8_0 && C <= 2 && SPLIT) {
    (void)q1;
    const uint32_t W[4] = {q0.x, q0.y, q0.z, q0.w};
    int I[C];
#pragma unroll
    for (int c = 0; c < C; ++c) I[c] = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t fl = W[i] ^ 0x88888888u;
      const uint32_t sel[2] = {W[i], W[i] >> 16}, self[2] = {fl, fl >> 16};
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const uint32_t lo = prmt(IQ4NL_LO_0, IQ4NL_LO_1, sel[h]);
        const uint32_t hi = prmt(IQ4NL_HIP1_0, IQ4NL_HIP1_1, self[h]);
#pragma unroll
        for (int c = 0; c < C; ++c) I[c] = dp4a(hi, act.a[c][2 * i + h], dp4a(lo, act.a[c][2 * i + h], I[c]));
      }
    }
#pragma unroll
    for (int c = 0; c < C; ++c) {
      if (I_out) I_out[c] = I[c];
      p[c] = __fmul_rn(__int2float_rn(I[c]), __fmul_rn(dw, act.d[c]));
    }
    return;
  }
  uint32_t wv[8];
  if constexpr (FMT == MOEX_Q8_0) {
    wv[0] = q0.x; wv[1] = q0.y; wv[2] = q0.z; wv[3] = q0.w;
    wv[4] = q1.x; wv[5] = q1.y; wv[6] = q1.z; wv[7] = q1.w;
  } else {
    (void)q1;
    const uint32_t W[4] = {q0.x, q0.y, q0.z, q0.w};
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

// Same, reading the block from memory at wq; with `swap` (Q8_0) the second
// 16-byte half first, for activations loaded with the same swap.
template <int FMT, int C>
__device__ __forceinline__ void block_row_dots(const uint8_t* wq, float dw, const ActRegs<FMT, C>& act, float* p,
                                               int* I_out = nullptr, bool swap = false) {
  const int o0 = swap ? 16 : 0;
  const uint4 q0 = *reinterpret_cast<const uint4*>(wq + o0);
  const uint4 q1 = FMT == MOEX_Q8_0 ? *reinterpret_cast<const uint4*>(wq + (16 - o0)) : q0;
  block_dots_from<FMT, C, true>(q0, q1, dw, act, p, I_out);
}

// Shared-memory reads of Q8_0 blocks: lane li of a half warp reads its
// 32-byte block at byte 32 * li of the row, so lanes li and li + 4 hit the
// same four banks.  Lanes with bit 2 set read the second half first; then
// lanes 0..7 cover all 32 banks and a half warp's 16-byte read takes two
// wavefronts instead of four (it costs a per-lane address, so it is used
// where shared-memory reads, not issue slots, bound the kernel).  Callers
// load their activations with the same swap.
template <int FMT>
__device__ __forceinline__ bool smem_half_swap(int li) {
  return FMT == MOEX_Q8_0 && ((li >> 2) & 1);
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

// The same sums without the two selects per exchanged pair.  Each lane keeps
// its values in the "xor layout": slot s holds logical value
// s ^ xor_layout_mask<N>(lane), i.e. lanes with bit 3 set hold the two
// halves swapped, lanes with bit 2 set the quarters inside them, and so on.
// Then at every level a lane sends slot i + N/2 and keeps slot i, and the
// pairs added are exactly those of halving_reduce, so both give the same
// bits and leave the results in the same lanes.
template <int N>
__device__ __forceinline__ int xor_layout_mask(int lane) {
  int m = 0;
  if constexpr (N >= 2) m |= ((lane >> 3) & 1) * (N / 2);
  if constexpr (N >= 4) m |= ((lane >> 2) & 1) * (N / 4);
  if constexpr (N >= 8) m |= ((lane >> 1) & 1) * (N / 8);
  if constexpr (N >= 16) m |= (lane & 1) * (N / 16);
  return m;
}

template <int N, int O>
__device__ __forceinline__ void halving_reduce_xl(float* v) {
  if constexpr (O > 0) {
    if constexpr (N > 1) {
#pragma unroll
      for (int i = 0; i < N / 2; ++i) v[i] = v[i] + __shfl_xor_sync(0xffffffffu, v[i + N / 2], O);
      halving_reduce_xl<N / 2, O / 2>(v);
    } else {
      v[0] = v[0] + __shfl_xor_sync(0xffffffffu, v[0], O);
      halving_reduce_xl<1, O / 2>(v);
    }
  }
}

// True when C values a lane can use the xor layout without padding slots:
// C is a power of two, so slot c holds column c ^ xor_layout_mask<C>(lane).
template <int C>
__host__ __device__ constexpr bool xor_layout_ok() { return (C & (C - 1)) == 0; }

// ----------------------------------------------------------------- consumer layout

// Warp w owns slice ks = w / WPS; its half `hf` (lane >> 4) and index
// jw = w % WPS give the stage rows jw*2 + hf + 2*WPS*i, i < RPH, with
// RPH = SR / (2*WPS).
struct ConsumerPos {
  int ks, jw, hf, li, lane, warp;
};

__device__ __forceinline__ ConsumerPos consumer_pos(int warp, int lane, int WPS) {
  ConsumerPos p;
  p.warp = warp;
  p.ks = warp / WPS;
  p.jw = warp % WPS;
  p.lane = lane;
  p.hf = lane >> 4;
  p.li = lane & 15;
  return p;
}

template <int C, int WPS, int N, typename Out>
__device__ __forceinline__ void reduce_out(float (&v)[N], const ConsumerPos& p, int nrows, Out&& out) {
  constexpr int RPH = SR / (2 * WPS);
  constexpr int V = RPH * C;
  halving_reduce<N, 8>(v, p.lane);
  const int li = p.li;
  if constexpr (N >= 16) {
#pragma unroll
    for (int i = 0; i < N / 16; ++i) {
      const int idx = li * (N / 16) + i;
      if (idx < V) {
        const int rr = idx / C, c = idx % C;
        const int row = p.jw * 2 + p.hf + 2 * WPS * rr;
        if (row < nrows) out(row, c, v[i]);
      }
    }
  } else {
    constexpr int REP = 16 / N;
    if (li % REP == 0) {
      const int idx = li / REP;
      if (idx < V) {
        const int rr = idx / C, c = idx % C;
        const int row = p.jw * 2 + p.hf + 2 * WPS * rr;
        if (row < nrows) out(row, c, v[0]);
      }
    }
  }
}

// reduce_out into red[row][ks][c].
template <int C, int WPS, int N>
__device__ __forceinline__ void reduce_to_red(float (&v)[N], const ConsumerPos& p, int nrows, int NS, float* red) {
  reduce_out<C, WPS, N>(v, p, nrows, [&](int row, int c, float val) { red[(row * NS + p.ks) * C + c] = val; });
}

template <int C, int WPS>
struct Vals {
  static constexpr int N = pow2_ceil((SR / (2 * WPS)) * C);
};

// Waits (bounded) until the red slot is free for stage `it`: its previous
// user (stage it - nred) has been summed.  Returns false on timeout / abort.
__device__ __forceinline__ bool red_slot_wait(volatile int* seq, int it, volatile int* abort) {
  if (*seq == it) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t i = 1;; ++i) {
    if (*seq == it) return true;
    if ((i & 63u) == 0) {
      if (abort && *abort) return false;
      if (global_timer_ns() - t0 > WAIT_LIMIT_NS) return false;
    }
  }
}

// K slices (of 16 blocks) of a row with NB blocks.
__host__ __device__ inline int num_slices(int NB) { return (NB + SLICE - 1) / SLICE; }

// ----------------------------------------------------------------- TMA ring

// A ring of shared-memory stages filled by one producer thread with bulk
// (TMA) copies of contiguous plane rows: slot = [SR rows x qrow bytes of
// quants][SR rows x scrow bytes of FP16 scales].  full[slot] completes when a
// stage's bytes have landed; empty[slot] when every consumer warp has let go.
struct TmaRing {
  uint64_t* full;
  uint64_t* empty;
  uint8_t* slots;
  int nst, slot_bytes, qrow, scrow;
  int slot_rows;  // row capacity of a slot (scales start at slot_rows * qrow)
  __device__ uint8_t* slot(int it) const { return slots + static_cast<size_t>(it % nst) * slot_bytes; }
};

// Producer side: waits for the slot of stage `it` to be free, then copies
// `nrows` rows starting at qsrc / ssrc.  Returns false on timeout / abort.
__device__ __forceinline__ bool tma_ring_fill(const TmaRing& R, int it, const uint8_t* qsrc, const uint8_t* ssrc,
                                              int nrows, uint64_t policy, volatile int* abort) {
  const int s = it % R.nst;
  if (it >= R.nst && !mbar_wait(&R.empty[s], ((it / R.nst) - 1) & 1, abort)) return false;
  uint8_t* dst = R.slots + static_cast<size_t>(s) * R.slot_bytes;
  mbar_arrive_expect_tx(&R.full[s], nrows * (R.qrow + R.scrow));
  bulk_g2s_stream(dst, qsrc, nrows * R.qrow, &R.full[s], policy);
  bulk_g2s_stream(dst + R.slot_rows * R.qrow, ssrc, nrows * R.scrow, &R.full[s], policy);
  return true;
}

// Consumer side: per-lane partial sums of 8 rows (rows row0 .. row0+nrows-1
// of the slot of ring stage `it`), after waiting for the slot to land when
// `wait` is set.  Returns false on timeout / abort.
// With SWAP, Q8_0 blocks are read with smem_half_swap and act must have been
// loaded with the same swap.
template <int FMT, int C, int WPS, int N, bool SWAP = false>
__device__ __forceinline__ bool tma_ring_partials(const TmaRing& R, int it, const ConsumerPos& p, int nrows, int NB,
                                                  const ActRegs<FMT, C>& act, float (&v)[N], volatile int* abort,
                                                  int row0 = 0, bool wait = true,
                                                  uint64_t limit_ns = WAIT_LIMIT_NS) {
#pragma unroll
  for (int i = 0; i < N; ++i) v[i] = 0.f;
  if (wait && !mbar_wait(&R.full[it % R.nst], (it / R.nst) & 1, abort, limit_ns)) return false;
  const uint8_t* st = R.slot(it) + row0 * R.qrow;
  const uint8_t* sc = R.slot(it) + R.slot_rows * R.qrow + row0 * R.scrow;
  const int b = p.ks * SLICE + p.li;
  if (b >= NB) return true;
  constexpr int RPH = SR / (2 * WPS);
  const bool swap = SWAP && smem_half_swap<FMT>(p.li);
#pragma unroll
  for (int rr = 0; rr < RPH; ++rr) {
    const int row = p.jw * 2 + p.hf + 2 * WPS * rr;
    if (row < nrows) {
      const uint8_t* wq = st + row * R.qrow + b * FmtTraits<FMT>::QBYTES;
      const float dw = __half2float(reinterpret_cast<const __half*>(sc + row * R.scrow)[b]);
      block_row_dots<FMT, C>(wq, dw, act, &v[rr * C], nullptr, swap);
    }
  }
  return true;
}

// Consumer side: this warp is done reading stage `it`'s slot.
__device__ __forceinline__ void tma_ring_release(const TmaRing& R, int it, int lane) {
  __syncwarp();
  if (lane == 0) mbar_arrive(&R.empty[it % R.nst]);
}

// Sum over the K slices (in slice order) of red[row][ks][c] for rows
// [row0, row0+nrows), spread over `nthreads` threads starting at `tid`.
template <int C, typename Out>
__device__ __forceinline__ void slices_final(const float* red, int row0, int nrows, int NS, int tid, int nthreads,
                                             Out&& out) {
  for (int idx = tid; idx < nrows * C; idx += nthreads) {
    const int row = row0 + idx / C, c = idx % C;
    float s = red[(row * NS + 0) * C + c];
    for (int ks = 1; ks < NS; ++ks) s = s + red[(row * NS + ks) * C + c];
    out(row, c, s);
  }
}

}  // namespace moex
