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
};

// Shared-memory carve-up of the dense GEMV (all offsets 16-byte aligned;
// stage slots 128-byte aligned).
struct GemvSmem {
  int bars, cnt, abort_flag, xs, xd, red, stages, total;
  __host__ __device__ GemvSmem(int C, int K, int NB, int NS, int nst, int stage_bytes) {
    int o = 0;
    bars = o; o += 16 * nst;
    cnt = o; o += 4 * nst;
    abort_flag = o; o += 16;
    o = (o + 15) & ~15;
    xs = o; o += C * K;
    o = (o + 15) & ~15;
    xd = o; o += 4 * C * NB;
    o = (o + 15) & ~15;
    red = o; o += 4 * nst * SR * NS * C;
    o = (o + 127) & ~127;
    stages = o; o += nst * stage_bytes;
    total = o;
  }
};

template <int FMT, int C, int WPS>
__global__ void __launch_bounds__(512, 1) qgemv_kernel(GemvArgs a) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const GemvSmem L(C, a.K, a.NB, a.NS, a.nst, a.stage_bytes);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bars);
  uint64_t* empty = full + a.nst;
  int* cnt = reinterpret_cast<int*>(smem + L.cnt);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L.abort_flag);
  int8_t* xs = reinterpret_cast<int8_t*>(smem + L.xs);
  float* xd = reinterpret_cast<float*>(smem + L.xd);
  float* red = reinterpret_cast<float*>(smem + L.red);
  uint8_t* stages = smem + L.stages;

  const int nwc = a.NS * WPS;  // consumer warps
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t G = gridDim.x;
  const int64_t row_begin = a.rows * blockIdx.x / G;
  const int64_t row_end = a.rows * (blockIdx.x + 1) / G;
  const int nstage = static_cast<int>((row_end - row_begin + SR - 1) / SR);

  if (threadIdx.x == 0) {
    for (int i = 0; i < a.nst; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], nwc);
      cnt[i] = 0;
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  pdl_launch_dependents();

  if (warp == nwc) {
    // ---------------- producer: stream the CTA's rows (weights only; they do
    // not depend on the previous kernel, so no griddepcontrol.wait here).
    if (lane == 0) {
      const uint64_t pol = l2_evict_first_policy();
      int issued = 0;
      for (int it = 0; it < nstage; ++it) {
        const int slot = it % a.nst;
        if (it >= a.nst && !mbar_wait(&empty[slot], ((it / a.nst) - 1) & 1, abort_flag)) {
          *abort_flag = 1;
          flag_status(a.status, DEV_TIMEOUT_PIPE);
          break;
        }
        const int64_t r0 = row_begin + static_cast<int64_t>(it) * SR;
        const int n = static_cast<int>((row_end - r0) < SR ? (row_end - r0) : SR);
        uint8_t* st = stages + static_cast<size_t>(slot) * a.stage_bytes;
        mbar_arrive_expect_tx(&full[slot], n * (a.qrow + a.scrow));
        bulk_g2s_stream(st, a.qs + r0 * a.qrow, n * a.qrow, &full[slot], pol);
        bulk_g2s_stream(st + SR * a.qrow, a.sc + r0 * a.scrow, n * a.scrow, &full[slot], pol);
        issued = it + 1;
      }
      // On abort, wait (bounded) for copies still landing in this CTA's smem.
      if (*abort_flag) {
        for (int it = max(0, issued - a.nst); it < issued; ++it)
          mbar_wait(&full[it % a.nst], (it / a.nst) & 1, nullptr);
      }
    }
    return;
  }

  // ---------------- consumers
  pdl_wait();  // activations come from the previous kernel
  {
    const int nthr = nwc * 32;
    const int4* src = reinterpret_cast<const int4*>(a.xq);
    int4* dst = reinterpret_cast<int4*>(xs);
    for (int i = threadIdx.x; i < C * a.K / 16; i += nthr) dst[i] = src[i];
    const float2* dsrc = reinterpret_cast<const float2*>(a.xds);
    for (int i = threadIdx.x; i < C * a.NB; i += nthr) xd[i] = dsrc[i].x;
    named_bar_sync(1, nthr);
  }
  ConsumerPos pos;
  pos.ks = warp / WPS;
  pos.jw = warp % WPS;
  pos.lane = lane;
  pos.hf = lane >> 4;
  pos.li = lane & 15;
  const int b = pos.ks * SLICE + pos.li;
  ActRegs<FMT, C> act;
  {
    const int8_t* xcol[C];
    const float* dcol[C];
#pragma unroll
    for (int c = 0; c < C; ++c) {
      xcol[c] = xs + c * a.K;
      dcol[c] = xd + c * a.NB;
    }
    load_act<FMT, C>(act, xcol, dcol, b, b < a.NB, pos.li);
  }

  for (int it = 0; it < nstage; ++it) {
    const int slot = it % a.nst;
    const bool ok = mbar_wait(&full[slot], (it / a.nst) & 1, abort_flag);
    if (!ok) {
      if (lane == 0) {
        *abort_flag = 1;
        flag_status(a.status, DEV_TIMEOUT_PIPE);
      }
      break;
    }
    const int64_t r0 = row_begin + static_cast<int64_t>(it) * SR;
    const int n = static_cast<int>((row_end - r0) < SR ? (row_end - r0) : SR);
    const uint8_t* st = stages + static_cast<size_t>(slot) * a.stage_bytes;
    float* rs = red + slot * (SR * a.NS * C);
    stage_partials<FMT, C, WPS>(st, st + SR * a.qrow, a.qrow, a.scrow, n, a.NB, a.NS, pos, act, rs);
    if (stage_arrive_last(&cnt[slot], nwc, lane)) {
      float* y = a.y;
      const int64_t ldy = a.ldy;
      stage_final<C>(rs, n, a.NS, lane, [&](int row, int c, float v) { y[c * ldy + r0 + row] = v; });
      if (lane == 0) cnt[slot] = 0;
      __syncwarp();
    }
    if (lane == 0) mbar_arrive(&empty[slot]);
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
  block_row_dots<FMT, 1>(qs + r * qrow + static_cast<int64_t>(b) * FmtTraits<FMT>::QBYTES, 1.f, act, li, &p, &I);
  dots[t] = I;
}

// ----------------------------------------------------------------- host side

namespace {

template <int FMT, int C, int WPS>
moex_status launch_one(const GemvArgs& base, int smem_cap, cudaStream_t s) {
  GemvArgs a = base;
  auto kern = qgemv_kernel<FMT, C, WPS>;
  // ring slots: as many as fit, at most 16
  const GemvSmem l0(C, a.K, a.NB, a.NS, 0, a.stage_bytes);
  int nst = (smem_cap - l0.total - 256) / (a.stage_bytes + 4 * SR * a.NS * C + 20);
  nst = nst > 16 ? 16 : nst;
  if (nst < 2) return MOEX_EUNSUPPORTED;
  a.nst = nst;
  const GemvSmem L(C, a.K, a.NB, a.NS, nst, a.stage_bytes);
  if (ensure_smem(reinterpret_cast<const void*>(kern), L.total) != cudaSuccess) return MOEX_ECUDA;
  const int64_t max_ctas = (a.rows + SR - 1) / SR;
  const int grid = static_cast<int>(max_ctas < sm_count() ? max_ctas : sm_count());
  const int threads = (a.NS * WPS + 1) * 32;
  return cuda_status(launch_pdl(kern, dim3(grid), dim3(threads), L.total, s, a));
}

template <int FMT, int C>
moex_status launch_c(const GemvArgs& a, int smem_cap, cudaStream_t s) {
  switch (warps_per_slice(a.NS)) {
    case 4: return launch_one<FMT, C, 4>(a, smem_cap, s);
    case 2: return launch_one<FMT, C, 2>(a, smem_cap, s);
    default: return launch_one<FMT, C, 1>(a, smem_cap, s);
  }
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
  if (a.NS * warps_per_slice(a.NS) > 15) return MOEX_EUNSUPPORTED;
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
