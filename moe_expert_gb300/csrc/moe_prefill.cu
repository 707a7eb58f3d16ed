// The grouped MoE prefill layer on FP16 tensor cores (tcgen05, sm_103a).
//
// What it computes (#2356 Summary: prompt rows sorted by expert, IQ4_NL
// weights dequantised to FP16 per tile for the tensor cores, FP32 sums;
// #1525 Change: each dequantised value one expression rounded by
// __float2half_rn, SwiGLU between the two products, the top-k combine):
//   order   = the (token, slot) entries sorted by expert, stable by entry
//   Xs[p]   = fp16(x[token(order[p])])                       (gather)
//   D1      = Wh_gu[e] . Xs^T over each expert's rows        (GEMM 1)
//   H[p]    = fp16(silu(g) * u)                              (GEMM 1 epilogue)
//   D2      = Wh_dn[e] . H^T                                 (GEMM 2)
//   out[t] += w[t, slot] * D2[., p]                          (GEMM 2 epilogue)
// with Wh = fp16_rn(fp32(d) * kvalues[idx]).
//
// GB300 design (not the pages' wmma kernels): the weights are the MMA's A
// operand and live in tensor memory: four warps dequantise 128 weight rows x
// 64 inputs per k-step straight from the IQ4_NL planes into TMEM with
// tcgen05.st (one thread per row, no shared-memory round trip); the sorted
// token rows are the B operand, 32-row boxes of a 2-D TMA tensor map with the
// 128-byte swizzle; one thread issues tcgen05.mma (M = 128, N = tile tokens
// rounded to 16, K = 16) into a double-buffered FP32 accumulator in TMEM, and
// four epilogue warps read it back with tcgen05.ld.  Because the token count
// of an expert is the MMA's N, ragged experts cost at most 15 padded columns
// per tile instead of a partial 128-row M tile.  CTAs run in clusters of two
// on the same token tile (neighbouring feature tiles): each loads half of the
// token boxes with TMA multicast into both, since one SM's TMA unit cannot
// feed an M = 128 MMA from L2 at full rate, and each CTA's MMA completion is
// committed to the release barriers of both.
//
// K order: every FP16 operand of the two GEMMs stores each 32-input block
// interleaved (position 2j = input j, 2j+1 = input j+16), the order in which
// an IQ4_NL block's index bytes hold them (low nibble j, high nibble j+16).
// The same permutation on both operands leaves every dot product unchanged.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "common.cuh"
#include "gemv_core.cuh"
#include "internal.h"
#include "tc.cuh"

namespace moex {

constexpr int PF_NMAX = 192;     // tokens per tile (MMA N), multiple of 16
constexpr int PF_BK = 64;        // inputs per k-step (one 128-byte swizzle row of FP16)
constexpr int PF_NB_ST = 4;      // B (token) stages in shared memory
constexpr int PF_BOXR = 32;      // token rows per TMA box
constexpr int PF_NA_ST = 4;      // A (weight) stages in TMEM
constexpr int PF_STAGE_B = PF_NMAX * PF_BK * 2;   // bytes of one B stage
constexpr int PF_ACOL = 2 * PF_NMAX;              // first TMEM column of the A stages
constexpr int PF_DQ_WARPS = 8;   // dequantising warps: two per TMEM lane quarter, one IQ4_NL block each
constexpr int PF_THREADS = (2 + PF_DQ_WARPS + 4) * 32;  // warp 0 TMA, 1 MMA + TMEM, dequant, 4 epilogue
constexpr int PF_EPI0 = 2 + PF_DQ_WARPS;                // first epilogue warp

// ----------------------------------------------------------------- sort

// counts[e] = number of entries routed to expert e (one CTA per expert).
__global__ void __launch_bounds__(256) prefill_count_kernel(const int32_t* __restrict__ ids, int n, int E,
                                                            int* __restrict__ counts, uint32_t* status) {
  pdl_wait();
  pdl_launch_dependents();
  const int e = blockIdx.x;
  int c = 0;
  for (int j = threadIdx.x; j < n; j += blockDim.x) {
    const int v = ids[j];
    c += v == e;
    if (e == 0 && (v < 0 || v >= E)) flag_status(status, DEV_BAD_ROUTE);
  }
  __shared__ int red[8];
  for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = c;
  __syncthreads();
  if (threadIdx.x == 0) {
    int s = 0;
    for (int i = 0; i < (int)(blockDim.x >> 5); ++i) s += red[i];
    counts[e] = s;
  }
}

struct PrefillTiles {
  int4* t1;     // GEMM 1 tiles {expert, feature tile, first row, rows}
  int4* t2;     // GEMM 2 tiles
  int* n1;      // number of GEMM 1 tiles
  int* n2;
  int F1, F2;   // feature tiles per expert (I/64, H/128)
};

__host__ __device__ inline int pf_token_tiles(int n) { return (n + PF_NMAX - 1) / PF_NMAX; }

// Stable placement (one CTA per expert): order[off_e + r] = the r-th entry
// (in entry order) routed to e; tokw[...] = {token, weight}; and the tiles
// of expert e for both GEMMs: ceil(n_e / 192) token tiles of balanced size,
// times the feature tiles.
__global__ void __launch_bounds__(256) prefill_place_kernel(const int32_t* __restrict__ ids, const float* __restrict__ w,
                                                            int n, int k, int E, const int* __restrict__ counts,
                                                            int* __restrict__ order, int2* __restrict__ tokw,
                                                            PrefillTiles tl) {
  pdl_wait();
  pdl_launch_dependents();
  const int e = blockIdx.x;
  __shared__ int s_off, s_tbase, s_wsum[8];
  if (threadIdx.x == 0) {
    int off = 0, tb = 0, tot = 0;
    for (int i = 0; i < E; ++i) {
      if (i < e) {
        off += counts[i];
        tb += pf_token_tiles(counts[i]);
      }
      tot += pf_token_tiles(counts[i]);
    }
    s_off = off;
    s_tbase = tb;
    if (e == E - 1) {
      *tl.n1 = tot * tl.F1;
      *tl.n2 = tot * tl.F2;
    }
  }
  __syncthreads();
  const int ne = counts[e];
  const int off = s_off;
  // tiles
  const int ntt = pf_token_tiles(ne);
  for (int i = threadIdx.x; i < ntt * tl.F1; i += blockDim.x) {
    const int tt = i / tl.F1, f = i % tl.F1;
    const int r0 = off + tt * ne / ntt, r1 = off + (tt + 1) * ne / ntt;
    tl.t1[(s_tbase + tt) * tl.F1 + f] = make_int4(e, f, r0, r1 - r0);
  }
  for (int i = threadIdx.x; i < ntt * tl.F2; i += blockDim.x) {
    const int tt = i / tl.F2, f = i % tl.F2;
    const int r0 = off + tt * ne / ntt, r1 = off + (tt + 1) * ne / ntt;
    tl.t2[(s_tbase + tt) * tl.F2 + f] = make_int4(e, f, r0, r1 - r0);
  }
  // stable compaction of the entries of expert e
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int base = 0;
  for (int j0 = 0; j0 < n; j0 += blockDim.x) {
    const int j = j0 + threadIdx.x;
    const bool mine = j < n && ids[j] == e;
    const unsigned bal = __ballot_sync(0xffffffffu, mine);
    if (lane == 0) s_wsum[warp] = __popc(bal);
    __syncthreads();
    int before = base;
    for (int i = 0; i < warp; ++i) before += s_wsum[i];
    if (mine) {
      const int r = before + __popc(bal & ((1u << lane) - 1u));
      order[off + r] = j;
      tokw[off + r] = make_int2(j / k, __float_as_int(w[j]));
    }
    int tot = 0;
    for (int i = 0; i < (int)(blockDim.x >> 5); ++i) tot += s_wsum[i];
    base += tot;
    __syncthreads();
  }
}

// ----------------------------------------------------------------- gather

// Xs[p] = fp16(x[token(order[p])]) with each 32-input block interleaved.
// One warp per sorted row; lane handles whole blocks.
__global__ void __launch_bounds__(256) prefill_gather_kernel(const uint16_t* __restrict__ x, int H, int k, int n,
                                                             const int* __restrict__ order, __half* __restrict__ xs) {
  pdl_wait();
  pdl_launch_dependents();
  const int row = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (row >= n) return;
  const int t = order[row] / k;
  const uint4* src = reinterpret_cast<const uint4*>(x + static_cast<int64_t>(t) * H);
  uint4* dst = reinterpret_cast<uint4*>(xs + static_cast<int64_t>(row) * H);
  for (int blk = lane; blk < H / QK; blk += 32) {
    uint32_t in[16];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint4 v = src[blk * 4 + i];
      in[4 * i] = v.x; in[4 * i + 1] = v.y; in[4 * i + 2] = v.z; in[4 * i + 3] = v.w;
    }
    // element e of the block: 16-bit half (e & 1) of word e >> 1
    auto elem = [&](int e) -> float {
      const uint32_t wv = in[e >> 1];
      const uint16_t b = (e & 1) ? static_cast<uint16_t>(wv >> 16) : static_cast<uint16_t>(wv & 0xFFFFu);
      return __uint_as_float(static_cast<uint32_t>(b) << 16);
    };
    uint32_t o[16];
#pragma unroll
    for (int jj = 0; jj < 16; ++jj) {
      const __half2 h = __halves2half2(__float2half_rn(elem(jj)), __float2half_rn(elem(jj + 16)));
      o[jj] = *reinterpret_cast<const uint32_t*>(&h);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) dst[blk * 4 + i] = make_uint4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]);
  }
}

// ----------------------------------------------------------------- GEMM

struct GemmArgs {
  const uint8_t* qs;   // IQ4_NL nibble plane of the weight stack
  const uint8_t* sc;   // FP16 scale plane
  int qrow, scrow;     // plane row strides (bytes)
  int64_t rows_per_expert;
  int K;               // inputs (hidden for GEMM 1, inter for GEMM 2)
  const int4* tiles;
  const int* ntiles;
  __half* Hs;          // GEMM 1 output [rows][I] (interleaved blocks)
  int I;
  float* out;          // GEMM 2 output [T][Hd]
  int Hd;
  const int2* tokw;    // per sorted row: token, weight bits
  uint32_t* status;
};

// The IQ4_NL codebook plus 128, as unsigned bytes: entries 0..7 (bit 7
// clear) and entries 8..15 with bit 7 cleared.
constexpr uint32_t IQ4B_LO_0 = 0x3F2D1801u;   // 1, 24, 45, 63
constexpr uint32_t IQ4B_LO_1 = 0x766A5D4Fu;   // 79, 93, 106, 118
constexpr uint32_t IQ4B_HI_0 = 0x26190D01u;   // 129, 141, 153, 166 & 0x7f
constexpr uint32_t IQ4B_HI_1 = 0x71594535u;   // 181, 197, 217, 241 & 0x7f

// kvalues[n] + 128 for the four indices in the low 16 bits of `sel`
// (selector nibble bit 3 flipped in `sel_flipped`): the low entries come
// from one prmt (zero where n >= 8), the high ones with bit 7 cleared from a
// second (zero where n < 8), and bit 7 is set where the high part is non-zero
// (every high entry has a non-zero low part).
__device__ __forceinline__ uint32_t iq4nl_biased4(uint32_t sel, uint32_t sel_flipped) {
  const uint32_t lo = prmt(IQ4B_LO_0, IQ4B_LO_1, sel);
  const uint32_t hi7 = prmt(IQ4B_HI_0, IQ4B_HI_1, sel_flipped);
  const uint32_t b7 = (hi7 + 0x7F7F7F7Fu) & 0x80808080u;
  return lo | hi7 | b7;
}

// Dequantises one IQ4_NL block (16 index bytes n, FP16 scale d) of one weight
// row into 16 TMEM column words: word j = half2(d * kv[lo(byte j)],
// d * kv[hi(byte j)]), each product rounded once to FP16 (an exact small
// integer times the FP16 scale, one HMUL2 rounding).  The integer is made
// exactly as FP16 from the biased byte u = kv + 128: the half with bits
// 0x6400 | u is 1024 + u, minus 1152.
__device__ __forceinline__ void dequant_block16(uint4 n, uint16_t dbits, uint32_t (&col)[16]) {
  const __half2 one152 = __half2half2(__ushort_as_half(0x6480));  // 1152
  const __half2 d2 = __half2half2(__ushort_as_half(dbits));
  const uint32_t W[4] = {n.x, n.y, n.z, n.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t wv = W[i];
    const uint32_t fl = wv ^ 0x88888888u;
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const uint32_t u = iq4nl_biased4(hh ? (wv >> 16) : wv, hh ? (fl >> 16) : fl);
      const uint32_t p0 = prmt(u, 0x64646464u, 0x4140u);  // half2(1024 + u0, 1024 + u1)
      const uint32_t p1 = prmt(u, 0x64646464u, 0x4342u);
      __half2 h0 = __hmul2(__hsub2(*reinterpret_cast<const __half2*>(&p0), one152), d2);
      __half2 h1 = __hmul2(__hsub2(*reinterpret_cast<const __half2*>(&p1), one152), d2);
      col[4 * i + 2 * hh] = *reinterpret_cast<uint32_t*>(&h0);
      col[4 * i + 2 * hh + 1] = *reinterpret_cast<uint32_t*>(&h1);
    }
  }
}

__device__ __forceinline__ uint4 ldg_nc_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}
__device__ __forceinline__ uint32_t ldg_nc_u32(const void* p) {
  uint32_t v;
  asm volatile("ld.global.nc.L1::no_allocate.u32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}

__device__ __forceinline__ void red_add_f32(float* p, float v) {
  asm volatile("red.global.add.f32 [%0], %1;" ::"l"(p), "f"(v) : "memory");
}

__device__ __forceinline__ int pf_mma_n(int nrows) { return (nrows + 15) & ~15; }

// Named barrier over `count` threads that also ORs a flag across them, so
// every participant takes the same branch afterwards.
__device__ __forceinline__ bool named_bar_or(uint32_t id, uint32_t count, bool flag) {
  uint32_t out;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.or.pred q, %2, %3, p;\n selp.u32 %0, 1, 0, q;\n}\n"
      : "=r"(out)
      : "r"(static_cast<uint32_t>(flag)), "r"(id), "r"(count)
      : "memory");
  return out != 0;
}

struct PfSmem {
  int b, bars, xbuf, tmem, abort_flag, total;
  __host__ __device__ PfSmem() {
    int o = 0;
    b = o; o += PF_NB_ST * PF_STAGE_B;                          // 1024-aligned (dynamic smem base)
    bars = o; o += 8 * (2 * PF_NB_ST + 2 * PF_NA_ST + 4 + 1);
    o = (o + 15) & ~15;
    xbuf = o; o += 2 * 32 * 33 * 4;
    tmem = o; o += 16;
    abort_flag = o; o += 16;
    total = o + 1024;                                          // slack for aligning the base
    if (total < 120 * 1024) total = 120 * 1024;                // one CTA per SM: it owns all 512 TMEM columns
  }
};

// EPI == 1: SwiGLU -> H (FP16).  EPI == 2: weighted combine into out.
// CL == 2: clusters of two CTAs sharing each token stage (multicast); CL == 1: alone.
template <int EPI, int CL>
__global__ void __launch_bounds__(PF_THREADS, 1) prefill_gemm_kernel(const __grid_constant__ CUtensorMap bmap,
                                                                     GemmArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const PfSmem L;
  uint8_t* sb = smem + L.b;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L.bars);
  uint64_t* b_full = bars;
  uint64_t* b_empty = b_full + PF_NB_ST;
  uint64_t* a_full = b_empty + PF_NB_ST;
  uint64_t* a_empty = a_full + PF_NA_ST;
  uint64_t* d_full = a_empty + PF_NA_ST;
  uint64_t* d_empty = d_full + 2;
  uint64_t* done_bar = d_empty + 2;
  float* xbuf = reinterpret_cast<float*>(smem + L.xbuf);
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + L.tmem);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L.abort_flag);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < PF_NB_ST; ++i) {
      mbar_init(&b_full[i], 1);
      mbar_init(&b_empty[i], CL);  // the MMAs of every CTA of the cluster
    }
    for (int i = 0; i < PF_NA_ST; ++i) {
      mbar_init(&a_full[i], PF_DQ_WARPS * 32);
      mbar_init(&a_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&d_full[i], 1);
      mbar_init(&d_empty[i], 128);
    }
    mbar_init(done_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&bmap);
  }
  if (warp == 1) {
    tmem_alloc(tmem_holder, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  if (CL == 2) cluster_sync_all();  // both CTAs' barriers are initialised before any multicast lands
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;

  pdl_wait();  // tiles, tokens and (GEMM 2) H come from earlier kernels
  pdl_launch_dependents();
  // tiles 2p and 2p+1 (same expert and tokens, neighbouring feature tiles)
  // go to the two CTAs of one cluster
  const int rank = CL == 2 ? static_cast<int>(cluster_ctarank()) : 0;
  const int t0 = CL == 2 ? 2 * (blockIdx.x >> 1) + rank : blockIdx.x;
  const int tstep = CL == 2 ? 2 * (gridDim.x >> 1) : gridDim.x;
  const int ntiles = *a.ntiles;
  const int KS = a.K / PF_BK;

  if (warp == 0) {
    // ------------------------------------------------ B producer (TMA)
    if (lane == 0) {
      int kc = 0;
      for (int t = t0; t < ntiles && !*abort_flag; t += tstep) {
        const int4 tile = a.tiles[t];
        const int nbox = (tile.w + PF_BOXR - 1) / PF_BOXR;
        for (int ks = 0; ks < KS; ++ks, ++kc) {
          const int s = kc % PF_NB_ST;
          if (kc >= PF_NB_ST && !mbar_wait(&b_empty[s], ((kc / PF_NB_ST) - 1) & 1, abort_flag)) {
            *abort_flag = 1;
            flag_status(a.status, DEV_TIMEOUT_MMA);
            break;
          }
          // the whole stage lands in this CTA (with CL == 2, half of the boxes from each CTA of the pair)
          mbar_arrive_expect_tx(&b_full[s], nbox * PF_BOXR * PF_BK * 2);
          for (int bx = rank; bx < nbox; bx += CL) {
            uint8_t* dst = sb + s * PF_STAGE_B + bx * PF_BOXR * PF_BK * 2;
            if (CL == 2)
              tma_load_2d_mc(dst, &bmap, ks * PF_BK, tile.z + PF_BOXR * bx, &b_full[s], 0x3);
            else
              tma_load_2d(dst, &bmap, ks * PF_BK, tile.z + PF_BOXR * bx, &b_full[s]);
          }
        }
      }
      // after an abort, let the copies already issued land before the CTA exits
      if (*abort_flag) {
        for (int j = kc - 1; j >= 0 && j >= kc - PF_NB_ST; --j)
          mbar_wait(&b_full[j % PF_NB_ST], (j / PF_NB_ST) & 1, nullptr);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer
    if (lane == 0) {
      int kc = 0, ti = 0;
      bool issued_any = false;
      for (int t = t0; t < ntiles && !*abort_flag; t += tstep, ++ti) {
        const int4 tile = a.tiles[t];
        const int ab = ti & 1;
        if (ti >= 2 && !mbar_wait(&d_empty[ab], ((ti >> 1) - 1) & 1, abort_flag)) {
          *abort_flag = 1;
          flag_status(a.status, DEV_TIMEOUT_MMA);
          break;
        }
        tc_fence_after();
        const uint32_t idesc = idesc_f16_f32(128, pf_mma_n(tile.w));
        const uint32_t dcol = tmem + ab * PF_NMAX;
        for (int ks = 0; ks < KS; ++ks, ++kc) {
          const int sa = kc % PF_NA_ST, sbk = kc % PF_NB_ST;
          if (!mbar_wait(&a_full[sa], (kc / PF_NA_ST) & 1, abort_flag) ||
              !mbar_wait(&b_full[sbk], (kc / PF_NB_ST) & 1, abort_flag)) {
            *abort_flag = 1;
            flag_status(a.status, DEV_TIMEOUT_MMA);
            break;
          }
          tc_fence_after();
          const uint32_t baddr = smem_u32(sb + sbk * PF_STAGE_B);
#pragma unroll
          for (int kk = 0; kk < PF_BK / 16; ++kk) {
            mma_f16_ts(dcol, tmem + PF_ACOL + sa * 32 + kk * 8, smem_desc_sw128(baddr + kk * 32), idesc,
                       (ks | kk) != 0);
          }
          issued_any = true;
          mma_commit(&a_empty[sa]);
          if (CL == 2)
            mma_commit_mc(&b_empty[sbk], 0x3);  // both CTAs' B stage is refilled once both MMAs are done
          else
            mma_commit(&b_empty[sbk]);
        }
        if (*abort_flag) break;
        mma_commit(&d_full[ab]);
      }
      // make sure no MMA is still running before the TMEM is released
      if (issued_any) {
        mma_commit(done_bar);
        mbar_wait(done_bar, 0, nullptr);
      }
    }
  } else if (warp < PF_EPI0) {
    // ------------------------------------------------ A producers: dequantise into TMEM
    // warp pair (w, w + 4) shares lane quarter q; half h dequantises block h
    // of each 64-input k-step (TMEM columns 16h .. 16h+15 of the stage).
    const int q = warp & 3;
    const int h = (warp - 2) >> 2;
    const int m = 32 * q + lane;  // A row = TMEM lane
    constexpr int PD = 3;         // k-steps of raw bytes in flight per thread
    int kc = 0;
    for (int t = t0; t < ntiles && !*abort_flag; t += tstep) {
      const int4 tile = a.tiles[t];
      int64_t row;
      if (EPI == 1) {
        const int64_t base = static_cast<int64_t>(tile.x) * a.rows_per_expert;
        row = m < 64 ? base + tile.y * 64 + m : base + a.I + tile.y * 64 + (m - 64);
      } else {
        row = static_cast<int64_t>(tile.x) * a.rows_per_expert + tile.y * 128 + m;
      }
      const uint8_t* qp = a.qs + row * a.qrow + 16 * h;
      const uint16_t* sp = reinterpret_cast<const uint16_t*>(a.sc + row * a.scrow) + h;
      uint4 rq[PD];
      uint16_t rs[PD];
#pragma unroll
      for (int i = 0; i < PD; ++i) {
        if (i < KS) {
          rq[i] = ldg_nc_v4(qp + i * 32);
          rs[i] = __ldg(sp + 2 * i);
        }
      }
      for (int ks = 0; ks < KS; ++ks, ++kc) {
        const uint4 cq = rq[0];
        const uint16_t cs = rs[0];
#pragma unroll
        for (int i = 0; i + 1 < PD; ++i) {
          rq[i] = rq[i + 1];
          rs[i] = rs[i + 1];
        }
        if (ks + PD < KS) {
          rq[PD - 1] = ldg_nc_v4(qp + (ks + PD) * 32);
          rs[PD - 1] = __ldg(sp + 2 * (ks + PD));
        }
        uint32_t col[16];
        dequant_block16(cq, cs, col);
        const int s = kc % PF_NA_ST;
        if (kc >= PF_NA_ST && !mbar_wait(&a_empty[s], ((kc / PF_NA_ST) - 1) & 1, abort_flag)) {
          *abort_flag = 1;
          flag_status(a.status, DEV_TIMEOUT_MMA);
          break;
        }
        tc_fence_after();
        tmem_st16(tmem + (static_cast<uint32_t>(32 * q) << 16) + PF_ACOL + s * 32 + 16 * h, col);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&a_full[s]);
      }
    }
  } else {
    // ------------------------------------------------ epilogue
    const int q = warp & 3;
    int ti = 0;
    for (int t = t0; t < ntiles; t += tstep, ++ti) {
      const int4 tile = a.tiles[t];
      const int ab = ti & 1;
      bool stop = *abort_flag != 0;
      if (!stop && !mbar_wait(&d_full[ab], (ti >> 1) & 1, abort_flag)) {
        *abort_flag = 1;
        flag_status(a.status, DEV_TIMEOUT_MMA);
        stop = true;
      }
      // the gate / up warp pair takes the same decision before its hand-offs
      if (EPI == 1) stop = named_bar_or(6 + (q & 1), 64, stop);
      if (stop) break;
      tc_fence_after();
      const uint32_t dbase = tmem + (static_cast<uint32_t>(32 * q) << 16) + ab * PF_NMAX;
      const int nchunk = (tile.w + 31) / 32;
      for (int c = 0; c < nchunk; ++c) {
        uint32_t r[32];
        tmem_ld32(dbase + 32 * c, r);
        tmem_ld_wait();
        if (EPI == 1) {
          const int pair = q & 1;
          float* xb = xbuf + pair * 32 * 33;
          if (q >= 2) {  // up rows: hand u to the gate warp of the same features
#pragma unroll
            for (int i = 0; i < 32; ++i) xb[lane * 33 + i] = __uint_as_float(r[i]);
            named_bar_sync(2 + pair, 64);
            named_bar_sync(4 + pair, 64);
          } else {
            named_bar_sync(2 + pair, 64);
            const int f = tile.y * 64 + 32 * q + lane;                   // intermediate index
            const int col = (f & ~31) + ((f & 31) < 16 ? 2 * (f & 15) : 2 * (f & 15) + 1);
            for (int i = 0; i < 32; ++i) {
              const int p = 32 * c + i;
              if (p < tile.w) {
                const float g = __uint_as_float(r[i]);
                const float u = xb[lane * 33 + i];
                const float h = __fmul_rn(__fdividef(g, 1.0f + __expf(-g)), u);
                a.Hs[static_cast<int64_t>(tile.z + p) * a.I + col] = __float2half_rn(h);
              }
            }
            named_bar_sync(4 + pair, 64);
          }
        } else {
          const int fo = tile.y * 128 + 32 * q + lane;   // output feature
          const int pl = 32 * c + lane;
          const int2 tw = pl < tile.w ? a.tokw[tile.z + pl] : make_int2(0, 0);
          for (int i = 0; i < 32; ++i) {
            const int tok = __shfl_sync(0xffffffffu, tw.x, i);
            const float wt = __int_as_float(__shfl_sync(0xffffffffu, tw.y, i));
            if (32 * c + i < tile.w) red_add_f32(a.out + static_cast<int64_t>(tok) * a.Hd + fo, wt * __uint_as_float(r[i]));
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&d_empty[ab]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (CL == 2) cluster_sync_all();  // no multicast copy or commit of the partner is still in flight
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ----------------------------------------------------------------- host side

namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

// 2-D FP16 map over [rows][cols] (row pitch cols*2 bytes), box 64 x PF_BOXR, 128-byte swizzle.
bool make_map(CUtensorMap* m, void* base, int64_t rows, int64_t cols) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols * 2)};
  const cuuint32_t box[2] = {PF_BK, PF_BOXR};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

using PfKernel = void (*)(CUtensorMap, GemmArgs);

cudaLaunchConfig_t pf_config(int grid, size_t smem, cudaStream_t s, int cl, cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(PF_THREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = cl;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cfg;
}

// Persistent grid: every CTA (cluster) resident at once.  For pairs this is
// twice the number of co-resident clusters, which can be below the SM count
// when a GPC has an odd number of free SMs.
int pf_grid(PfKernel kern, int cl, size_t smem) {
  if (cl == 1) return sm_count();
  static int cached[2] = {0, 0};
  static PfKernel which[2] = {nullptr, nullptr};
  for (int i = 0; i < 2; ++i)
    if (which[i] == kern) return cached[i];
  cudaLaunchAttribute attr[2];
  cudaLaunchConfig_t cfg = pf_config(sm_count(), smem, nullptr, cl, attr);
  int nclusters = 0;
  if (cudaOccupancyMaxActiveClusters(&nclusters, kern, &cfg) != cudaSuccess || nclusters <= 0) {
    cudaGetLastError();
    nclusters = sm_count() / 2;
  }
  const int slot = which[0] == nullptr ? 0 : 1;
  which[slot] = kern;
  cached[slot] = 2 * nclusters;
  return cached[slot];
}

cudaError_t launch_pf_gemm(PfKernel kern, int cl, size_t smem, cudaStream_t s, const CUtensorMap& map,
                           const GemmArgs& args) {
  cudaLaunchAttribute attr[2];
  cudaLaunchConfig_t cfg = pf_config(pf_grid(kern, cl, smem), smem, s, cl, attr);
  return cudaLaunchKernelEx(&cfg, kern, map, args);
}

}  // namespace

// Workspace layout (offsets in bytes, each 256-aligned).
void prefill_ws_layout(int T, int k, int E, int64_t hidden, int64_t inter, size_t* off) {
  const size_t n = static_cast<size_t>(T) * k;
  const size_t tiles = n / PF_NMAX + E + 1;
  size_t o = 0;
  off[0] = o; o = align_up(o + 4 * E, 256);                              // counts
  off[1] = o; o = align_up(o + 4 * n, 256);                              // order
  off[2] = o; o = align_up(o + 8 * n, 256);                              // tokw
  off[3] = o; o = align_up(o + 16 * tiles * (inter / 64), 256);          // tiles 1
  off[4] = o; o = align_up(o + 16 * tiles * (hidden / 128), 256);        // tiles 2
  off[5] = o; o = align_up(o + 16, 256);                                 // n1, n2
  off[6] = o; o = align_up(o + 2 * n * hidden, 256);                     // Xs
  off[7] = o; o = align_up(o + 2 * n * inter, 256);                      // Hs
  off[8] = o;                                                            // total
}

size_t moe_prefill_ws_bytes(int T, int k, int E, int64_t hidden, int64_t inter) {
  size_t off[9];
  prefill_ws_layout(T, k, E, hidden, inter, off);
  return off[8];
}

moex_status launch_moe_prefill(const moex_qweight* gu, const moex_qweight* dn, const uint16_t* x, int T,
                               const int32_t* ids, const float* w, int k, float* out, void* ws, cudaStream_t s) {
  const int E = gu->n_mats;
  const int H = static_cast<int>(gu->K), I = static_cast<int>(dn->K);
  const int n = T * k;
  size_t off[9];
  prefill_ws_layout(T, k, E, H, I, off);
  uint8_t* wsb = static_cast<uint8_t*>(ws);
  int* counts = reinterpret_cast<int*>(wsb + off[0]);
  int* order = reinterpret_cast<int*>(wsb + off[1]);
  int2* tokw = reinterpret_cast<int2*>(wsb + off[2]);
  PrefillTiles tl;
  tl.t1 = reinterpret_cast<int4*>(wsb + off[3]);
  tl.t2 = reinterpret_cast<int4*>(wsb + off[4]);
  tl.n1 = reinterpret_cast<int*>(wsb + off[5]);
  tl.n2 = tl.n1 + 1;
  tl.F1 = I / 64;
  tl.F2 = H / 128;
  __half* xs = reinterpret_cast<__half*>(wsb + off[6]);
  __half* hs = reinterpret_cast<__half*>(wsb + off[7]);
  uint32_t* status = device_status_ptr();

  CUtensorMap m1, m2;
  if (!make_map(&m1, xs, n, H) || !make_map(&m2, hs, n, I)) return MOEX_ECUDA;

  if (launch_pdl(prefill_count_kernel, dim3(E), dim3(256), 0, s, ids, n, E, counts, status) != cudaSuccess)
    return MOEX_ECUDA;
  if (launch_pdl(prefill_place_kernel, dim3(E), dim3(256), 0, s, ids, w, n, k, E, static_cast<const int*>(counts),
                 order, tokw, tl) != cudaSuccess)
    return MOEX_ECUDA;
  if (launch_pdl(prefill_gather_kernel, dim3((n * 32 + 255) / 256), dim3(256), 0, s, x, H, k, n,
                 static_cast<const int*>(order), xs) != cudaSuccess)
    return MOEX_ECUDA;
  const PfSmem L;
  // pairs share each token stage when both GEMMs have an even number of feature tiles
  const int cl = (tl.F1 % 2 == 0 && tl.F2 % 2 == 0) ? 2 : 1;
  const PfKernel k1 = cl == 2 ? prefill_gemm_kernel<1, 2> : prefill_gemm_kernel<1, 1>;
  const PfKernel k2 = cl == 2 ? prefill_gemm_kernel<2, 2> : prefill_gemm_kernel<2, 1>;
  if (ensure_smem(reinterpret_cast<const void*>(k1), L.total) != cudaSuccess ||
      ensure_smem(reinterpret_cast<const void*>(k2), L.total) != cudaSuccess)
    return MOEX_ECUDA;
  GemmArgs g1 = {};
  g1.qs = static_cast<const uint8_t*>(gu->qs);
  g1.sc = static_cast<const uint8_t*>(gu->scales);
  g1.qrow = static_cast<int>(qs_row_bytes(gu->fmt, gu->K));
  g1.scrow = static_cast<int>(sc_row_bytes(gu->K));
  g1.rows_per_expert = gu->rows;
  g1.K = H;
  g1.tiles = tl.t1;
  g1.ntiles = tl.n1;
  g1.Hs = hs;
  g1.I = I;
  g1.status = status;
  if (launch_pf_gemm(k1, cl, L.total, s, m1, g1) != cudaSuccess) return MOEX_ECUDA;
  if (cudaMemsetAsync(out, 0, static_cast<size_t>(T) * H * sizeof(float), s) != cudaSuccess) return MOEX_ECUDA;
  GemmArgs g2 = {};
  g2.qs = static_cast<const uint8_t*>(dn->qs);
  g2.sc = static_cast<const uint8_t*>(dn->scales);
  g2.qrow = static_cast<int>(qs_row_bytes(dn->fmt, dn->K));
  g2.scrow = static_cast<int>(sc_row_bytes(dn->K));
  g2.rows_per_expert = dn->rows;
  g2.K = I;
  g2.tiles = tl.t2;
  g2.ntiles = tl.n2;
  g2.out = out;
  g2.Hd = H;
  g2.tokw = tokw;
  g2.status = status;
  if (launch_pf_gemm(k2, cl, L.total, s, m2, g2) != cudaSuccess) return MOEX_ECUDA;
  return MOEX_OK;
}

}  // namespace moex
