// Dense multi-column GEMV: Q8_0 or IQ4_NL weights x q8_1 activations,
// 1..8 columns per pass (#242 What it does; #1424 What changed).
#include <cuda_fp16.h>

#include <mutex>

#include "common.cuh"
#include "gemv_core.cuh"
#include "internal.h"

namespace moex {

struct GemvArgs {
  const uint8_t* qs;    // quant plane
  const uint8_t* sc;    // scale plane
  int64_t rows;
  int K, NB, NS;        // inputs, blocks, K slices
  int qrow, scrow;      // plane row strides (bytes)
  int nst;              // ring slots
  int stage_bytes;      // bytes of one ring slot
  const int8_t* xq;     // q8_1 quants [ncols][K]
  const float* xds;     // {d, s} [ncols][NB]
  float* y;
  int64_t ldy;
  uint32_t* status;
  uint64_t wait_ns;     // limit of every bounded wait (WAIT_LIMIT_NS)
  int starve;           // test hook: the ring producer issues no copies
};



constexpr int GEMV_CHUNK = 8;  // stages whose slice partials are summed together

// Shared-memory carve-up of the dense ring GEMV.
struct GemvSmem {
  int bars, cnt, abort_flag, red, ring, total;
  __host__ __device__ GemvSmem(int C, int NS, int nst, int slot_bytes) {
    int o = 0;
    bars = o; o += 16 * nst;
    cnt = o; o += 4 * nst;
    abort_flag = o; o += 16;
    o = (o + 15) & ~15;
    red = o; o += 4 * GEMV_CHUNK * SR * NS * C;
    o = (o + 127) & ~127;
    ring = o; o += nst * slot_bytes;
    total = o;
  }
};

// Threads of a dense ring GEMV CTA: NS*WPS*CS consumer warps + 1 producer
// warp (CS column groups, each warp computing C/CS of the columns).
// MINB == 2 variants keep registers and shared memory small enough that a
// CTA of the next GEMV in the stream can be resident beside this one, so
// with programmatic dependent launch its weight stream starts while this
// one drains.
template <int WPS, int MINB, int CS>
struct GemvBounds {
  static constexpr int MAXT = MINB == 2 ? (5 * WPS * CS + 1) * 32
                                        : ((5 * WPS * CS + 1) * 32 > 512 ? (5 * WPS * CS + 1) * 32 : 512);
};

// Ring variant: every CTA owns a contiguous range of rows; one producer
// thread streams them through a shared-memory ring with bulk (TMA) copies,
// starting before griddepcontrol.wait (the weights do not depend on the
// previous kernel); the consumer warps load their activation blocks straight
// into registers after the wait.  The partial sums of a stage are reduced
// over the half warp into a per-chunk buffer; every GEMV_CHUNK stages the
// consumers meet at a barrier and sum over the K slices (no per-stage
// hand-off between warps).
template <int FMT, int C, int WPS, int MINB, int CS>
__global__ void __launch_bounds__(GemvBounds<WPS, MINB, CS>::MAXT, MINB) qgemv_kernel(GemvArgs a) {
  static_assert(C % CS == 0, "column groups split the columns evenly");
  constexpr int CG = C / CS;  // columns of one consumer warp
  extern __shared__ __align__(1024) uint8_t smem[];
  MOEX_TRACE_BEGIN();
  const int nwc = a.NS * WPS * CS;
  const int slot_bytes = a.stage_bytes;
  const GemvSmem L(C, a.NS, a.nst, slot_bytes);
  TmaRing R;
  R.full = reinterpret_cast<uint64_t*>(smem + L.bars);
  R.empty = R.full + a.nst;
  R.slots = smem + L.ring;
  R.nst = a.nst;
  R.slot_bytes = slot_bytes;
  R.qrow = a.qrow;
  R.scrow = a.scrow;
  R.slot_rows = SR;
  int* cnt = reinterpret_cast<int*>(smem + L.cnt);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L.abort_flag);
  float* red = reinterpret_cast<float*>(smem + L.red);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t G = gridDim.x;
  const int64_t row_begin = a.rows * blockIdx.x / G;
  const int64_t row_end = a.rows * (blockIdx.x + 1) / G;
  const int nstage = static_cast<int>((row_end - row_begin + SR - 1) / SR);
  auto stage_rows = [&](int it) {
    const int64_t r0 = row_begin + static_cast<int64_t>(it) * SR;
    return static_cast<int>((row_end - r0) < SR ? (row_end - r0) : SR);
  };

  if (threadIdx.x == 0) {
    for (int i = 0; i < a.nst; ++i) {
      mbar_init(&R.full[i], 1);
      mbar_init(&R.empty[i], nwc);
      cnt[i] = 0;
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  MOEX_TRACE_STAMP(0);
  pdl_launch_dependents();

  if (warp == nwc) {
    if (lane == 0 && !a.starve) {
      const uint64_t pol = l2_evict_first_policy();
      int issued = 0;
      for (int it = 0; it < nstage; ++it) {
        const int64_t r0 = row_begin + static_cast<int64_t>(it) * SR;
        if (!tma_ring_fill(R, it, a.qs + r0 * a.qrow, a.sc + r0 * a.scrow, stage_rows(it), pol, abort_flag)) {
          *abort_flag = 1;
          flag_status(a.status, DEV_TIMEOUT_PIPE);
          break;
        }
        issued = it + 1;
      }
      // On abort, wait (bounded) for copies still landing in this CTA's smem.
      if (*abort_flag)
        for (int it = max(0, issued - a.nst); it < issued; ++it) mbar_wait(&R.full[it % a.nst], (it / a.nst) & 1, nullptr);
    }
    return;
  }

  const int cg = warp / (a.NS * WPS);  // column group: columns cg*CG .. cg*CG+CG-1
  const ConsumerPos pos = consumer_pos(warp % (a.NS * WPS), lane, WPS);
  pdl_wait();  // activations come from the previous kernel
  MOEX_TRACE_STAMP(1);
  ActRegs<FMT, CG> act;
  {
    const int8_t* xcol[CG];
    const float* dcol[CG];
#pragma unroll
    for (int c = 0; c < CG; ++c) {
      xcol[c] = a.xq + static_cast<int64_t>(cg * CG + c) * a.K;
      dcol[c] = a.xds + static_cast<int64_t>(cg * CG + c) * a.NB * 2;
    }
    const int b = pos.ks * SLICE + pos.li;
    load_act<FMT, CG>(act, xcol, dcol, b, b < a.NB, pos.li, 2);
  }
  constexpr int N = Vals<CG, WPS>::N;
  const int nthr = nwc * 32;
  bool dead = false;
  for (int c0 = 0; c0 < nstage; c0 += GEMV_CHUNK) {
    const int c1 = min(c0 + GEMV_CHUNK, nstage);
    for (int it = c0; it < c1 && !dead; ++it) {
      const int n = stage_rows(it);
      float v[N];
      if (!tma_ring_partials<FMT, CG, WPS, N>(R, it, pos, n, a.NB, act, v, abort_flag, 0, true, a.wait_ns)) {
        if (lane == 0) {
          *abort_flag = 1;
          flag_status(a.status, DEV_TIMEOUT_PIPE);
        }
        dead = true;
        break;
      }
      float* rs = red + (it - c0) * (SR * a.NS * C);
      const int NS = a.NS;
      reduce_out<CG, WPS, N>(v, pos, n, [&](int row, int c, float val) { rs[(row * NS + pos.ks) * C + cg * CG + c] = val; });
      tma_ring_release(R, it, lane);
    }
    named_bar_sync(1, nthr);
    if (!dead) {
      const int64_t r0 = row_begin + static_cast<int64_t>(c0) * SR;
      const int64_t span = static_cast<int64_t>(c1 - c0) * SR;
      const int nrows = static_cast<int>(span < row_end - r0 ? span : row_end - r0);
      float* y = a.y;
      const int64_t ldy = a.ldy;
      slices_final<C>(red, 0, nrows, a.NS, threadIdx.x, nthr,
                      [&](int row, int c, float val) { y[c * ldy + r0 + row] = val; });
    }
    named_bar_sync(1, nthr);
  }
  MOEX_TRACE_STAMP(2);
}

// ----------------------------------------------------------------- register-staged GEMV

// Small-column variant: every lane streams its CTA's weight bytes through
// registers with plain 16-byte ld.global.nc, P stages ahead; the first P
// stages are issued before griddepcontrol.wait, so they are in flight while
// the previous kernel finishes; nothing waits for ring slots or the TMA
// unit.  With MINB == 2 the kernel fits in half an SM (<= 48 registers a
// thread), so the next GEMV in the stream is resident beside it and its
// first stages load while this one drains.  Four warps per K slice, one row
// per half warp per 8-row stage.  Partial sums are reduced over the half
// warp and then over the slices, in slice order, exactly as in the ring
// variant (same tree: same bits).
constexpr int REG_WPS = 4;

template <int FMT, int C, int NSTG, int P, int MINB>
__global__ void __launch_bounds__(640, MINB) qgemv_reg_kernel(GemvArgs a) {
  extern __shared__ __align__(16) uint8_t smem[];
  float* red = reinterpret_cast<float*>(smem);  // [NSTG*8 rows][NS][C]
  constexpr int QB16 = FmtTraits<FMT>::QBYTES / 16;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const ConsumerPos pos = consumer_pos(warp, lane, REG_WPS);
  const int64_t G = gridDim.x;
  const int64_t row_begin = a.rows * blockIdx.x / G;
  const int64_t row_end = a.rows * (blockIdx.x + 1) / G;
  const int nrows = static_cast<int>(row_end - row_begin);
  const int b = pos.ks * SLICE + pos.li;
  const bool bvalid = b < a.NB;
  const int my_row0 = pos.jw * 2 + pos.hf;  // row within each stage

  uint4 q[P][QB16];
  uint32_t sw[P];
  auto load_stage = [&](int st, int slot) {
    const int row = st * SR + my_row0;
    if (bvalid && row < nrows) {
      const uint8_t* src = a.qs + (row_begin + row) * a.qrow + b * FmtTraits<FMT>::QBYTES;
#pragma unroll
      for (int h = 0; h < QB16; ++h)
        asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                     : "=r"(q[slot][h].x), "=r"(q[slot][h].y), "=r"(q[slot][h].z), "=r"(q[slot][h].w)
                     : "l"(src + 16 * h));
      asm volatile("ld.global.nc.L1::no_allocate.u32 %0, [%1];"
                   : "=r"(sw[slot])
                   : "l"(a.sc + (row_begin + row) * a.scrow + 4 * (b >> 1)));
    } else {
#pragma unroll
      for (int h = 0; h < QB16; ++h) q[slot][h] = make_uint4(0, 0, 0, 0);
      sw[slot] = 0;
    }
  };
#pragma unroll
  for (int st = 0; st < P; ++st)
    if (st < NSTG) load_stage(st, st);
  pdl_launch_dependents();
  pdl_wait();  // activations come from the previous kernel
  constexpr int N = pow2_ceil(C);
  constexpr bool XL = xor_layout_ok<C>();  // partial sums in the xor layout (select-free reduce)
  const int cmask = XL ? xor_layout_mask<N>(lane) : 0;
  ActRegs<FMT, C> act;
  {
    const int8_t* xcol[C];
    const float* dcol[C];
#pragma unroll
    for (int c = 0; c < C; ++c) {
      xcol[c] = a.xq + static_cast<int64_t>(c ^ cmask) * a.K;
      dcol[c] = a.xds + static_cast<int64_t>(c ^ cmask) * a.NB * 2;
    }
    load_act<FMT, C>(act, xcol, dcol, b, bvalid, pos.li, 2);
  }
#pragma unroll
  for (int st = 0; st < NSTG; ++st) {
    const int slot = st % P;
    const int row = st * SR + my_row0;
    float v[N];
#pragma unroll
    for (int i = 0; i < N; ++i) v[i] = 0.f;
    if (bvalid && row < nrows) {
      const uint16_t hb = static_cast<uint16_t>((b & 1) ? (sw[slot] >> 16) : (sw[slot] & 0xFFFFu));
      block_dots_from<FMT, C>(q[slot][0], q[slot][QB16 - 1], __half2float(__ushort_as_half(hb)), act, v);
    }
    if (st + P < NSTG) load_stage(st + P, slot);  // refill the slot just consumed
    if constexpr (XL)
      halving_reduce_xl<N, 8>(v);
    else
      halving_reduce<N, 8>(v, lane);
    // lane li holds value li / (16/N) (N < 16 always here)
    constexpr int REP = 16 / N;
    if (pos.li % REP == 0) {
      const int c = pos.li / REP;
      if (c < C && row < nrows) red[(row * a.NS + pos.ks) * C + c] = v[0];
    }
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < nrows * C; idx += blockDim.x) {
    const int row = idx / C, c = idx % C;
    float s = red[(row * a.NS + 0) * C + c];
    for (int ks = 1; ks < a.NS; ++ks) s = s + red[(row * a.NS + ks) * C + c];
    a.y[c * a.ldy + row_begin + row] = s;
  }
}

// Diagnostic kernel: per-block integer dots with the GEMV's own device code.
template <int FMT>
__global__ void block_dots_kernel(const uint8_t* __restrict__ qs, int64_t rows, int K, int NB, int qrow,
                                  const int8_t* __restrict__ xq, int ncols, int32_t* __restrict__ dots) {
  const int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t total = static_cast<int64_t>(ncols) * rows * NB;
  if (t >= total) return;
  const int b = static_cast<int>(t % NB);
  const int64_t r = (t / NB) % rows;
  const int c = static_cast<int>(t / (static_cast<int64_t>(NB) * rows));
  const int li = threadIdx.x & 15;  // any lane position gives the same integer chain
  ActRegs<FMT, 1> act;
  const int8_t* xcol[1] = {xq + static_cast<int64_t>(c) * K};
  load_act<FMT, 1>(act, xcol, nullptr, b, true, li);
  float p;
  int I;
  block_row_dots<FMT, 1>(qs + r * qrow + static_cast<int64_t>(b) * FmtTraits<FMT>::QBYTES, 1.f, act, &p, &I);
  dots[t] = I;
}

// ----------------------------------------------------------------- host side

namespace {

template <int FMT, int C, int WPS, int MINB, int CS = 1>
moex_status launch_one(const GemvArgs& base, int smem_cap, cudaStream_t s) {
  GemvArgs a = base;
  auto kern = qgemv_kernel<FMT, C, WPS, MINB, CS>;
  // ring slots: as many as fit the budget (two CTAs per SM for MINB == 2), at most 8
  const int budget = MINB == 2 ? 110 * 1024 : smem_cap;
  const int slot_bytes = ((SR * (a.qrow + a.scrow)) + 127) & ~127;
  a.stage_bytes = slot_bytes;
  int nst = 8;
  for (; nst >= 2; --nst)
    if (GemvSmem(C, a.NS, nst, slot_bytes).total <= budget) break;
  if (nst < 2) return MOEX_EUNSUPPORTED;
  a.nst = nst;
  const GemvSmem L(C, a.NS, nst, slot_bytes);
  if (ensure_smem(reinterpret_cast<const void*>(kern), L.total) != cudaSuccess) return MOEX_ECUDA;
  const int64_t max_ctas = (a.rows + SR - 1) / SR;
  const int grid = static_cast<int>(max_ctas < sm_count() ? max_ctas : sm_count());
  const int threads = (a.NS * WPS * CS + 1) * 32;
  return cuda_status(launch_pdl(kern, dim3(grid), dim3(threads), L.total, s, a));
}

// Register-staged variant: K <= 2560 (5 slices x 4 warps = 640 threads), the
// CTA's rows fit NSTG stages, and the columns are few enough that the
// weights, scales and activations all fit the register budget.
template <int FMT, int C, int NSTG, int P, int MINB>
moex_status launch_reg(const GemvArgs& a, cudaStream_t s) {
  auto kern = qgemv_reg_kernel<FMT, C, NSTG, P, MINB>;
  const int64_t cap_rows = static_cast<int64_t>(SR) * NSTG;
  int64_t grid = sm_count();
  if ((a.rows + grid - 1) / grid > cap_rows) grid = (a.rows + cap_rows - 1) / cap_rows;
  if (grid > a.rows) grid = a.rows;
  const int smem = 4 * NSTG * SR * a.NS * C;
  if (ensure_smem(reinterpret_cast<const void*>(kern), smem) != cudaSuccess) return MOEX_ECUDA;
  const int threads = a.NS * REG_WPS * 32;
  return cuda_status(launch_pdl(kern, dim3(static_cast<unsigned>(grid)), dim3(threads), smem, s, a));
}

// Consumer layout: for K up to 2560 (<= 5 slices) two warps per slice for
// <= 4 columns, one for more (register budget of two resident CTAs); for
// larger K one warp per slice and one CTA per SM.
template <int FMT, int C>
moex_status launch_c(const GemvArgs& a, int smem_cap, cudaStream_t s) {
  if constexpr (C <= 4) {
    // register-staged, P stages ahead: one column streams 3 (IQ4_NL 4)
    // stages ahead at two CTAs per SM; two columns keep every stage in
    // flight; three and four columns stream 4 (IQ4_NL 6) ahead, one CTA per SM
    constexpr int NSTG = FMT == MOEX_IQ4_NL ? 12 : 8;
    constexpr bool HALF = C == 1;
    constexpr int P = HALF ? (FMT == MOEX_Q8_0 ? 3 : 4) : C <= 2 ? NSTG : (FMT == MOEX_Q8_0 ? 4 : 6);
    if (a.NS <= 5 && a.rows <= static_cast<int64_t>(sm_count()) * SR * NSTG * 4)
      return launch_reg<FMT, C, NSTG, P, HALF ? 2 : 1>(a, s);
  }
  if (a.NS <= 5) {
    // (K beyond the register-staged limits) up to 4 columns: two warps per
    // slice, two CTAs per SM (the next GEMV overlaps this one's drain); more
    // columns are compute-bound: one CTA per SM with twice the warps, the
    // columns split over two warp groups
    // (IQ4_NL keeps one column group: a second would decode every block twice)
    if constexpr (C <= 4) return launch_one<FMT, C, 2, 2>(a, smem_cap, s);
    else if constexpr (C % 2 == 0 && FMT == MOEX_Q8_0) return launch_one<FMT, C, 2, 1, 2>(a, smem_cap, s);
    else return launch_one<FMT, C, 2, 1>(a, smem_cap, s);
  }
  return launch_one<FMT, C, 1, 1>(a, smem_cap, s);
}

template <int FMT>
moex_status launch_fmt(const GemvArgs& a, int C, int smem_cap, cudaStream_t s) {
  switch (C) {
    case 1: return launch_c<FMT, 1>(a, smem_cap, s);
    case 2: return launch_c<FMT, 2>(a, smem_cap, s);
    case 3: return launch_c<FMT, 3>(a, smem_cap, s);
    case 4: return launch_c<FMT, 4>(a, smem_cap, s);
    case 5: return launch_c<FMT, 5>(a, smem_cap, s);
    case 6: return launch_c<FMT, 6>(a, smem_cap, s);
    case 7: return launch_c<FMT, 7>(a, smem_cap, s);
    default: return launch_c<FMT, 8>(a, smem_cap, s);
  }
}

}  // namespace

moex_status launch_qgemv(const moex_qweight* W, const int8_t* xq, const float* xds, int ncols, float* y,
                         int64_t ldy, cudaStream_t s) {
  GemvArgs a = {};
  a.qs = static_cast<const uint8_t*>(W->qs);
  a.sc = static_cast<const uint8_t*>(W->scales);
  a.rows = W->rows;
  a.K = static_cast<int>(W->K);
  a.NB = a.K / QK;
  a.NS = num_slices(a.NB);
  a.qrow = static_cast<int>(qs_row_bytes(W->fmt, W->K));
  a.scrow = static_cast<int>(sc_row_bytes(W->K));
  a.stage_bytes = ((SR * (a.qrow + a.scrow)) + 127) & ~127;
  a.status = device_status_ptr();
  a.wait_ns = WAIT_LIMIT_NS;
  a.starve = 0;
  if (a.NS > 16) return MOEX_EUNSUPPORTED;
  const int cap = max_smem_optin();
  for (int c0 = 0; c0 < ncols; c0 += 8) {
    const int C = ncols - c0 < 8 ? ncols - c0 : 8;
    a.xq = xq + static_cast<int64_t>(c0) * a.K;
    a.xds = xds + static_cast<int64_t>(c0) * a.NB * 2;
    a.y = y + static_cast<int64_t>(c0) * ldy;
    a.ldy = ldy;
    const moex_status st = W->fmt == MOEX_Q8_0 ? launch_fmt<MOEX_Q8_0>(a, C, cap, s)
                                               : launch_fmt<MOEX_IQ4_NL>(a, C, cap, s);
    if (st != MOEX_OK) return st;
  }
  return MOEX_OK;
}

moex_status launch_qgemv_starved(const moex_qweight* W, const int8_t* xq, const float* xds, int ncols, float* y,
                                 int64_t ldy, uint64_t wait_ns, cudaStream_t s) {
  GemvArgs a = {};
  a.qs = static_cast<const uint8_t*>(W->qs);
  a.sc = static_cast<const uint8_t*>(W->scales);
  a.rows = W->rows;
  a.K = static_cast<int>(W->K);
  a.NB = a.K / QK;
  a.NS = num_slices(a.NB);
  a.qrow = static_cast<int>(qs_row_bytes(W->fmt, W->K));
  a.scrow = static_cast<int>(sc_row_bytes(W->K));
  a.status = device_status_ptr();
  a.wait_ns = wait_ns;
  a.starve = 1;
  a.xq = xq;
  a.xds = xds;
  a.y = y;
  a.ldy = ldy;
  if (a.NS > 5) return MOEX_EUNSUPPORTED;
  // the ring variant of the one-column GEMV (the register-staged kernel has no producer)
  const int cap = max_smem_optin();
  (void)ncols;
  return W->fmt == MOEX_Q8_0 ? launch_one<MOEX_Q8_0, 1, 2, 2>(a, cap, s) : launch_one<MOEX_IQ4_NL, 1, 2, 2>(a, cap, s);
}

moex_status launch_block_dots(const moex_qweight* W, const int8_t* xq, int ncols, int32_t* dots, cudaStream_t s) {
  const int K = static_cast<int>(W->K), NB = K / QK;
  const int64_t total = static_cast<int64_t>(ncols) * W->rows * NB;
  const unsigned grid = static_cast<unsigned>((total + 127) / 128);
  const int qrow = static_cast<int>(qs_row_bytes(W->fmt, W->K));
  if (W->fmt == MOEX_Q8_0)
    block_dots_kernel<MOEX_Q8_0><<<grid, 128, 0, s>>>(static_cast<const uint8_t*>(W->qs), W->rows, K, NB, qrow, xq,
                                                      ncols, dots);
  else
    block_dots_kernel<MOEX_IQ4_NL><<<grid, 128, 0, s>>>(static_cast<const uint8_t*>(W->qs), W->rows, K, NB, qrow,
                                                        xq, ncols, dots);
  return cuda_status(cudaGetLastError());
}

}  // namespace moex
