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
// operand and live in tensor memory: eight warps dequantise 128 weight rows x
// 128 inputs per k-step straight from the IQ4_NL (or Q8_0) planes into TMEM
// with tcgen05.st (one thread per row, no shared-memory round trip); the
// sorted token rows are the B operand, boxes of a 2-D TMA tensor map with the
// 128-byte swizzle; tcgen05.mma (K = 16, N = tile tokens rounded up) into a
// double-buffered FP32 accumulator in TMEM, read back by eight epilogue warps
// with tcgen05.ld.  Because the token count of an expert is the MMA's N,
// a ragged expert costs at most 15 padded columns (its tiles are multiples
// of 16 rows but the last) instead of a partial 128-row M tile.  CTAs run in pairs (clusters of two) on neighbouring
// feature tiles of the same token tile and share M = 256 MMAs (tcgen05
// cta_group::2): each CTA loads only its half of the token rows, so the
// shared-memory traffic of the B operand per SM is halved.
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

constexpr int PF_SUBN = 192;     // tokens of one MMA sub-tile (one TMEM accumulator slot)
constexpr int PF_CAP_PAIR = 384; // tokens of a tile for CTA pairs: two sub-tiles
constexpr int PF_CAP_ONE = 192;  // tokens of a tile for single CTAs: one sub-tile
constexpr int PF_BK = 128;       // inputs per k-step (two 128-byte swizzle rows of FP16); K's last may be 64
constexpr int PF_BOXK = 64;      // inputs per token-row TMA box (one 128-byte swizzle row)
constexpr int PF_B_BYTES = 3 * 2 * 192 * 64 * 2;  // shared memory of the B (token) stages: 144 KB
constexpr int PF_NB_MAX = 6;     // most B stages (CTAs of a MoE pair: 96 rows, 24 KB a stage)
constexpr int PF_NA_ST = 2;      // A (weight) stages in TMEM
constexpr int PF_KD = 6;         // k-step-done barriers: k-step kc's MMAs commit to kdone[kc % 6]
static_assert(PF_KD % PF_NA_ST == 0, "a k-step's stages free on its own barrier");

// Token rows a CTA holds of a tile: 96 for a CTA of a MoE pair (tiles of at
// most 192 rows, one sub-tile), 192 otherwise (one CTA; or the dense pair's
// two sub-tiles of up to 96 rows each).  The B stages take PF_B_BYTES: six
// stages of 24 KB or three of 48 KB.
template <int EPI, bool PAIR>
__host__ __device__ constexpr int pf_rows_cta() { return PAIR && EPI != 3 ? 96 : 192; }
constexpr int PF_ACOL = 2 * PF_SUBN;              // first TMEM column of the A stages (after two slots)
constexpr int PF_ACOLS = PF_BK / 2;               // TMEM columns of one A stage (FP16 pairs)
static_assert(PF_ACOL + PF_NA_ST * PF_ACOLS <= 512, "accumulators and A stages fit the TMEM");
constexpr int PF_DQ_WARPS = 8;   // dequantising warps: two per TMEM lane quarter, one IQ4_NL block each
constexpr int PF_DQ0 = 3;        // first dequantising warp
constexpr int PF_EPI0 = PF_DQ0 + PF_DQ_WARPS;           // first epilogue warp
constexpr int PF_EPI_WARPS = 8;  // epilogue warps: two per TMEM lane quarter, alternate 32-column chunks
constexpr int PF_THREADS = (PF_EPI0 + PF_EPI_WARPS) * 32;  // warp 0 B TMA, 1 MMA + TMEM, 2 A TMA, dequant, epilogue
// Raw weight stages: the IQ4_NL bytes of 128 rows x 4 k-steps (8 blocks a
// row), two boxes of 64 rows x 128 bytes with the 128-byte swizzle, then
// their FP16 scales, two boxes of 64 rows x 16 bytes.
constexpr int PF_RAW_KS = 2;                      // k-steps per IQ4_NL raw stage (Q8_0: 1, same bytes)
constexpr int PF_NR_ST = 4;                       // raw stages
constexpr int PF_RAW_QS = 128 * 128;              // nibble bytes of a raw stage
constexpr int PF_RAW_STAGE = PF_RAW_QS + 128 * 16;  // + scale bytes (multiple of 1024)
__host__ __device__ constexpr int pf_raw_ks(int wf) { return wf == MOEX_Q8_0 ? 1 : PF_RAW_KS; }

// ----------------------------------------------------------------- sort

// Stable counting sort of the T*k entries by expert in three launches:
// per-segment histograms, one CTA that scans them (expert offsets, segment
// bases, tile lists), and a per-segment scatter that ranks equal experts
// in entry order with warp match.  Entries whose id is out of range are
// flagged and left out (the later kernels only see placed rows).

struct PrefillTiles {
  int4* t1;     // GEMM 1 tiles {expert, feature tile, first row, rows}
  int4* t2;     // GEMM 2 tiles
  int* n1;      // number of GEMM 1 tiles; n1[1] GEMM 2 tiles, n1[2] placed rows
  int* n2;
  int F1, F2;   // feature tiles per expert (I/64, H/128)
  int cap;      // most token rows a tile takes (PF_CAP_ONE for the MoE layer)
};

// An expert's n rows are cut into ceil(n / cap) token tiles of balanced size
// (the first n % nt tiles one row longer), so every tile of an expert does
// about the same MMA work per dequantised weight stage.
// Token tiles of n rows with at most cap rows (a multiple of 16) each: the
// fewest tiles, all but the last of the same size, that size a multiple of
// 16 (the MMA's N granularity), so the padding of a whole expert is under 16
// rows rather than under 16 rows a tile.
__host__ __device__ inline int pf_tile_rows(int n, int cap) {
  const int nt = (n + cap - 1) / cap;
  return (((n + nt - 1) / nt) + 15) & ~15;
}
__host__ __device__ inline int pf_token_tiles(int n, int cap) {
  if (n <= 0) return 0;
  const int b = pf_tile_rows(n, cap);
  return (n + b - 1) / b;
}
__host__ __device__ inline void pf_tile_span(int n, int cap, int t, int* r0, int* rows) {
  const int b = pf_tile_rows(n, cap);
  *r0 = t * b;
  *rows = n - t * b < b ? n - t * b : b;
}

constexpr int PF_MAX_SEGS = 1024;   // at most this many histogram segments

// Entries per segment: a multiple of 32, at least 256, at most PF_MAX_SEGS segments.
__host__ __device__ inline int pf_seg_len(int n) {
  int seg = (n + PF_MAX_SEGS - 1) / PF_MAX_SEGS;
  seg = seg < 256 ? 256 : seg;
  return (seg + 31) & ~31;
}
__host__ __device__ inline int pf_nsegs(int n) { return (n + pf_seg_len(n) - 1) / pf_seg_len(n); }

// hist[s][e] = entries of segment s routed to e (one CTA per segment).
__global__ void __launch_bounds__(256) prefill_hist_kernel(const int32_t* __restrict__ ids, int n, int E,
                                                           int* __restrict__ hist, uint32_t* status) {
  extern __shared__ int h_s[];
  pdl_wait();
  pdl_launch_dependents();
  for (int e = threadIdx.x; e < E; e += blockDim.x) h_s[e] = 0;
  __syncthreads();
  const int seg = pf_seg_len(n);
  const int j0 = blockIdx.x * seg, j1 = min(n, j0 + seg);
  for (int j = j0 + threadIdx.x; j < j1; j += blockDim.x) {
    const int v = ids[j];
    if (v < 0 || v >= E)
      flag_status(status, DEV_BAD_ROUTE);
    else
      atomicAdd(&h_s[v], 1);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) hist[static_cast<int64_t>(blockIdx.x) * E + e] = h_s[e];
}

// Exclusive scan of v over the block (blockDim.x == 1024); returns the total.
__device__ __forceinline__ int block_exscan(int& v, int* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) red[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int t = red[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, t, o);
      if (lane >= o) t += y;
    }
    red[lane] = t;
  }
  __syncthreads();
  const int total = red[31];
  v = x - v + (warp ? red[warp - 1] : 0);
  __syncthreads();
  return total;
}

// One CTA of 1024 threads, thread i owns experts 4i .. 4i+3 (E <= 4096):
// counts, first sorted row eoff[e] and first token tile etb[e] of each
// expert (etb[E] = all token tiles), hist[s][e] -> first sorted row of
// segment s's entries for e, and the totals n1[0..3] = GEMM 1 tiles,
// GEMM 2 tiles, placed rows, token tiles.
__global__ void __launch_bounds__(1024) prefill_scan_kernel(int n, int E, int* __restrict__ hist,
                                                            int* __restrict__ counts, int* __restrict__ eoff,
                                                            int* __restrict__ etb, PrefillTiles tl) {
  __shared__ int red[32];
  __shared__ int part[1024];    // [segment group][expert]: partial counts, then their exclusive prefix
  __shared__ int eoff_s[512];
  pdl_wait();
  pdl_launch_dependents();
  const int S = pf_nsegs(n);
  if (E <= 512) {
    // G groups of segments per expert, one thread each (a warp reads 32
    // experts of one segment: coalesced)
    const int G = 1024 / E;
    const int t = threadIdx.x, e = t % E, gr = t / E;
    const int s0 = gr < G ? S * gr / G : 0, s1 = gr < G ? S * (gr + 1) / G : 0;
    int v = 0;
    for (int sg = s0; sg < s1; ++sg) v += hist[static_cast<int64_t>(sg) * E + e];
    if (gr < G) part[gr * E + e] = v;
    __syncthreads();
    int c = 0, tiles = 0;
    if (t < E) {
      for (int g = 0; g < G; ++g) {  // the groups' exclusive prefix, in segment order
        const int x = part[g * E + t];
        part[g * E + t] = c;
        c += x;
      }
      tiles = pf_token_tiles(c, tl.cap);
    }
    int off = c, tb = tiles;
    const int placed = block_exscan(off, red);
    const int ttot = block_exscan(tb, red);
    if (t == 0) {
      tl.n1[0] = ttot * tl.F1;
      tl.n1[1] = ttot * tl.F2;
      tl.n1[2] = placed;
      tl.n1[3] = ttot;
      etb[E] = ttot;
    }
    if (t < E) {
      counts[t] = c;
      eoff[t] = off;
      etb[t] = tb;
      eoff_s[t] = off;
    }
    __syncthreads();
    // hist[s][e] becomes the first sorted row of segment s's entries of e
    if (gr < G) {
      int run = eoff_s[e] + part[gr * E + e];
      for (int sg = s0; sg < s1; ++sg) {
        int* hp = hist + static_cast<int64_t>(sg) * E + e;
        const int h = *hp;
        *hp = run;
        run += h;
      }
    }
    return;
  }
  // more experts: four a thread, segments in series
  int c[4];
  int csum = 0, tsum = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int e = 4 * threadIdx.x + i;
    int v = 0;
    if (e < E)
      for (int sg = 0; sg < S; ++sg) v += hist[static_cast<int64_t>(sg) * E + e];
    c[i] = v;
    csum += v;
    tsum += pf_token_tiles(v, tl.cap);
  }
  int off = csum, tb = tsum;
  const int placed = block_exscan(off, red);
  const int ttot = block_exscan(tb, red);
  if (threadIdx.x == 0) {
    tl.n1[0] = ttot * tl.F1;
    tl.n1[1] = ttot * tl.F2;
    tl.n1[2] = placed;
    tl.n1[3] = ttot;
    etb[E] = ttot;
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int e = 4 * threadIdx.x + i;
    if (e >= E) break;
    counts[e] = c[i];
    eoff[e] = off;
    etb[e] = tb;
    int run = off;
    for (int sg = 0; sg < S; ++sg) {
      int* hp = hist + static_cast<int64_t>(sg) * E + e;
      const int h = *hp;
      *hp = run;
      run += h;
    }
    off += c[i];
    tb += pf_token_tiles(c[i], tl.cap);
  }
}

// Both tile lists, one thread per tile: token tile g belongs to the last
// expert e with etb[e] <= g; its token tiles (pf_tile_span) cut the
// expert's rows into tiles of a multiple of 16 rows.  etb[0..E] is staged in shared memory (E + 1 ints)
// for the binary search.
__global__ void __launch_bounds__(256) prefill_tiles_kernel(int E, const int* __restrict__ counts,
                                                            const int* __restrict__ eoff, const int* __restrict__ etb,
                                                            PrefillTiles tl) {
  extern __shared__ int etb_s[];
  pdl_wait();
  pdl_launch_dependents();
  for (int e = threadIdx.x; e <= E; e += blockDim.x) etb_s[e] = etb[e];
  __syncthreads();
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t TT = tl.n1[3];
  const bool first = i < TT * tl.F1;
  const int64_t j = first ? i : i - TT * tl.F1;
  const int F = first ? tl.F1 : tl.F2;
  if (j >= TT * F) return;
  const int g = static_cast<int>(j / F), f = static_cast<int>(j % F);
  int lo = 0, hi = E;  // first e with etb[e] > g is in (lo, hi]
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (etb_s[mid] <= g) lo = mid; else hi = mid - 1;
  }
  const int e = lo;
  int r0, rows;
  pf_tile_span(counts[e], tl.cap, g - etb[e], &r0, &rows);
  (first ? tl.t1 : tl.t2)[j] = make_int4(e, f, eoff[e] + r0, rows);
}

// Dense product: token tiles (pf_tile_span) of at most `cap` rows times feature
// tiles of 128 rows, all of matrix 0; n1[0] = tiles, n1[2] = rows.
__global__ void __launch_bounds__(256) dense_tiles_kernel(int T, int F, int cap, int4* __restrict__ tiles,
                                                          int* __restrict__ n1) {
  pdl_wait();
  pdl_launch_dependents();
  const int ntt = pf_token_tiles(T, cap);
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i == 0) {
    n1[0] = ntt * F;
    n1[1] = 0;
    n1[2] = T;
    n1[3] = ntt;
  }
  if (i >= ntt * F) return;
  const int tt = i / F, f = i % F;
  int r0, rows;
  pf_tile_span(T, cap, tt, &r0, &rows);
  tiles[i] = make_int4(0, f, r0, rows);
}

// One warp per segment, entries in order, 32 at a time: equal experts are
// ranked by lane with __match_any_sync; order[row] = entry, pos[entry] = row
// (-1 for an entry left out), tokw[row] =
// {token, weight bits}.
__global__ void __launch_bounds__(32) prefill_scatter_kernel(const int32_t* __restrict__ ids,
                                                             const float* __restrict__ w, int n, int k, int E,
                                                             const int* __restrict__ hist, int* __restrict__ order,
                                                             int2* __restrict__ tokw, int* __restrict__ pos) {
  extern __shared__ int run[];
  pdl_wait();
  pdl_launch_dependents();
  const int lane = threadIdx.x;
  for (int e = lane; e < E; e += 32) run[e] = hist[static_cast<int64_t>(blockIdx.x) * E + e];
  __syncwarp();
  const int seg = pf_seg_len(n);
  const int j0 = blockIdx.x * seg, j1 = min(n, j0 + seg);
  constexpr int SC = 8;  // 32-entry steps whose ids and weights are loaded up front
  for (int jc = j0; jc < j1; jc += 32 * SC) {
    int vv[SC];
    float wv[SC];
#pragma unroll
    for (int u = 0; u < SC; ++u) {
      const int j = jc + 32 * u + lane;
      vv[u] = j < j1 ? ids[j] : -1;
      wv[u] = j < j1 ? w[j] : 0.f;
    }
#pragma unroll
    for (int u = 0; u < SC; ++u) {
      const int j = jc + 32 * u + lane;
      const int v = vv[u];
      const bool ok = v >= 0 && v < E;
      const unsigned peers = __match_any_sync(0xffffffffu, ok ? v : -1);
      int row = -1;
      if (ok) {
        row = run[v] + __popc(peers & ((1u << lane) - 1u));
        order[row] = j;
        tokw[row] = make_int2(j / k, __float_as_int(wv[u]));
      }
      if (j < j1) pos[j] = row;
      __syncwarp();
      // the highest lane of each group advances the expert's next row
      if (ok && (peers >> lane) == 1u) run[v] += __popc(peers);
      __syncwarp();
    }
  }
}

// ----------------------------------------------------------------- gather

// Xs[pos[t*k+s]] = fp16(x[t]) for every entry (t, s) placed by the sort
// (pos[] < 0: left out; pos == nullptr: the dense product, row t), with each
// 32-input block interleaved (FP16 word j of a block holds inputs j and
// j + 16).  One warp per token, in token order, so each input row is read
// from memory once and written to its k sorted rows.  Lane l takes 16-byte
// quarters q of the row's blocks (quarter index 4 * block + q = l, l + 32,
// ...), so a warp's stores cover 512 contiguous bytes; a quarter's inputs
// are the two 8-byte runs 4q..4q+3 and 16+4q..19+4q of the block.  Given
// out_vec4 > 0 (the integer route), the same threads initialise the layer
// output, which the down product accumulates into: zeros, or the residual
// when one is given (which may be out itself).  In the FP16 route the first
// GEMM's epilogue warps do that instead, under its MMAs.
__global__ void __launch_bounds__(256) prefill_gather_kernel(const uint16_t* __restrict__ x, int H, int T, int k,
                                                             const int* __restrict__ pos, __half* __restrict__ xs,
                                                             const float4* res, float4* out, int64_t out_vec4) {
  constexpr int CH = 4;  // quarters a lane converts before its k rows of stores
  pdl_wait();
  pdl_launch_dependents();
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t nthreads = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t z = i; z < out_vec4; z += nthreads) out[z] = res ? res[z] : make_float4(0.f, 0.f, 0.f, 0.f);
  const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (t >= T) return;
  const int lane = threadIdx.x & 31;
  int myrow = -1;  // lane s < k: the sorted row of entry (t, s)
  if (pos) {
    if (lane < k) myrow = pos[static_cast<int64_t>(t) * k + lane];
  } else if (lane == 0) {
    myrow = t;
  }
  const int nq = 4 * (H / QK);
  const uint2* src = reinterpret_cast<const uint2*>(x + static_cast<int64_t>(t) * H);
  for (int q0 = 0; q0 < nq; q0 += 32 * CH) {
    uint4 o[CH];
#pragma unroll
    for (int c = 0; c < CH; ++c) {
      const int qi = q0 + 32 * c + lane;
      if (qi >= nq) break;
      const int q = qi & 3;
      const uint2 lo = __ldg(src + 2 * (qi - q) + q), hi = __ldg(src + 2 * (qi - q) + 4 + q);
      // a BF16 is the upper half of an FP32; each FP16 pair (4q + j, 16 + 4q + j)
      // is one round-to-nearest conversion of two FP32s, the first in the low half
      const uint32_t a[4] = {lo.x << 16, lo.x & 0xFFFF0000u, lo.y << 16, lo.y & 0xFFFF0000u};
      const uint32_t b[4] = {hi.x << 16, hi.x & 0xFFFF0000u, hi.y << 16, hi.y & 0xFFFF0000u};
      uint32_t w[4];
#pragma unroll
      for (int j = 0; j < 4; ++j)
        asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(w[j]) : "f"(__uint_as_float(b[j])), "f"(__uint_as_float(a[j])));
      o[c] = make_uint4(w[0], w[1], w[2], w[3]);
    }
    for (int sl = 0; sl < k; ++sl) {
      const int row = __shfl_sync(0xffffffffu, myrow, sl);
      if (row < 0) continue;
      uint4* dst = reinterpret_cast<uint4*>(xs + static_cast<int64_t>(row) * H);
#pragma unroll
      for (int c = 0; c < CH; ++c) {
        const int qi = q0 + 32 * c + lane;
        if (qi < nq) dst[qi] = o[c];
      }
    }
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
  int8_t* Hq;          // integer route: q8_1 quants of H [rows][I] (natural order)
  float2* Hds;         // integer route: {d, s} of each 32-feature block [rows][I/32]
  float* Hf;           // integer route, optional: FP32 H [rows][I] (natural order)
  int I;
  float* out;          // GEMM 2 output [T][Hd]
  int Hd;
  const int2* tokw;    // per sorted row: token, weight bits
  // GEMM 1 of the FP16 route: the layer output the second GEMM accumulates
  // into, initialised to init_res (or zeros) as init_vec4 float4s, each CTA
  // a contiguous slice, a piece after each of its tiles
  float4* init_out;
  const float4* init_res;
  int64_t init_vec4;
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

// Dequantises one Q8_0 block (32 int8 q in two 16-byte halves lo = q[0..15],
// hi = q[16..31], FP16 scale d) into the same 16 TMEM column words as
// dequant_block16: word j = half2(d * q[j], d * q[j+16]), each product
// rounded once to FP16.  The byte q + 128 becomes the FP16 1024 + q + 128
// exactly (0x6400 | byte), minus 1152 gives q.
__device__ __forceinline__ void dequant_q8_block16(uint4 lo, uint4 hi, uint16_t dbits, uint32_t (&col)[16]) {
  const __half2 one152 = __half2half2(__ushort_as_half(0x6480));  // 1152
  const __half2 d2 = __half2half2(__ushort_as_half(dbits));
  const uint32_t L[4] = {lo.x, lo.y, lo.z, lo.w}, H[4] = {hi.x, hi.y, hi.z, hi.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    // [q4i, q4i+16, q4i+1, q4i+17] and [q4i+2, q4i+18, q4i+3, q4i+19], biased by 128
    const uint32_t u01 = prmt(L[i], H[i], 0x5140u) ^ 0x80808080u;
    const uint32_t u23 = prmt(L[i], H[i], 0x7362u) ^ 0x80808080u;
    const uint32_t U[2] = {u01, u23};
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const uint32_t p0 = prmt(U[hh], 0x64646464u, 0x4140u);
      const uint32_t p1 = prmt(U[hh], 0x64646464u, 0x4342u);
      __half2 h0 = __hmul2(__hsub2(*reinterpret_cast<const __half2*>(&p0), one152), d2);
      __half2 h1 = __hmul2(__hsub2(*reinterpret_cast<const __half2*>(&p1), one152), d2);
      col[4 * i + 2 * hh] = *reinterpret_cast<uint32_t*>(&h0);
      col[4 * i + 2 * hh + 1] = *reinterpret_cast<uint32_t*>(&h1);
    }
  }
}

__device__ __forceinline__ void red_add_f32(float* p, float v) {
  asm volatile("red.global.add.f32 [%0], %1;" ::"l"(p), "f"(v) : "memory");
}


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
  int b, raw, bars, xch, tmem, abort_flag, total;
  __host__ __device__ PfSmem() {
    int o = 0;
    b = o; o += PF_B_BYTES;                                     // 1024-aligned (dynamic smem base)
    raw = o; o += PF_NR_ST * PF_RAW_STAGE;                      // 1024-aligned
    bars = o; o += 8 * (PF_NB_MAX + PF_KD + PF_NA_ST + 2 * PF_NR_ST + 4 + 1);  // b_full, kdone, full, d_full/d_empty, done, r_full/r_empty
    o = (o + 15) & ~15;
    xch = o; o += 4 * 2 * 2 * 32 * 4;                          // integer route: per warp pair, amax and sums of 32 columns
    tmem = o; o += 16;
    abort_flag = o; o += 16;
    total = o + 1024;                                          // slack for aligning the base
    if (total < 120 * 1024) total = 120 * 1024;                // one CTA per SM: it owns all 512 TMEM columns
  }
};

// Token rows per TMA box: all the rows a CTA holds of a sub-tile, 96 for a
// CTA of a pair (half of at most 192), 192 for one CTA, so a k-step's token
// rows are one box per 64-input half and sub-tile (large boxes move L2-resident
// rows at about 1.4x the rate of 32-row boxes; rows past a short tile are
// loaded and not used).
template <bool PAIR>
__host__ __device__ constexpr int pf_boxr() { return PAIR ? 96 : 192; }

// MMA N of a sub-tile of `nrows` tokens: a multiple of 16 (for a pair each
// CTA holds N/2 rows, a multiple of 8: whole 8-row swizzle atoms).
template <bool PAIR>
__device__ __forceinline__ int pf_mma_n(int nrows) { return (nrows + 15) & ~15; }

// How a tile of `rows` tokens is laid out: sub-tile h (h = 0, 1) covers tile
// rows [start[h], start[h] + rows[h]) with MMA width n[h] into TMEM slot h
// (columns h * PF_SUBN ..); in a B stage this CTA's rows of sub-tile h start
// at row off[h] and take nbox[h] TMA boxes.  A pair's even CTA holds rows
// [0, n/2) of each sub-tile and the odd CTA rows [n/2, n).
template <bool PAIR>
struct PfSubTiles {
  int start[2], rows[2], n[2], off[2], nbox[2];
  __device__ __forceinline__ PfSubTiles(int tile_rows) {
    constexpr int BOXR = pf_boxr<PAIR>();
    // one sub-tile up to PF_SUBN rows, else two of about half the rows (the
    // first a multiple of 32, at most PF_SUBN), so neither MMA is narrow
    const int half = (((tile_rows + 1) / 2) + 31) & ~31;
    rows[0] = tile_rows <= PF_SUBN ? tile_rows : (half < PF_SUBN ? half : PF_SUBN);
    rows[1] = tile_rows - rows[0];
    start[0] = 0;
    start[1] = rows[0];
    off[0] = 0;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      n[h] = rows[h] > 0 ? pf_mma_n<PAIR>(rows[h]) : 0;
      const int held = PAIR ? n[h] / 2 : rows[h];
      nbox[h] = (held + BOXR - 1) / BOXR;
    }
    off[1] = nbox[0] * BOXR;
  }
};

// Feature tile row of TMEM lane m in GEMM 1 (rows 0..63 gate, 64..127 up in
// the raw weight stage).  The lanes of warp q hold, for 16 features j of a
// 32-feature block and the 16 features j + 16 of the same block, the gate
// row (lane bit 3 clear) and the up row (bit 3 set): gate and up of a
// feature are lanes l and l ^ 8, features j and j + 16 lanes l and l ^ 16.
__device__ __forceinline__ int pf_gu_feature(int m) {
  const int q = m >> 5, l = m & 31;
  return 32 * (q >> 1) + 8 * (q & 1) + (l & 7) + 16 * (l >> 4);
}
__device__ __forceinline__ int pf_gu_raw_row(int m) {
  return ((m >> 3) & 1) * 64 + pf_gu_feature(m);
}

// EPI == 1: SwiGLU -> H (FP16).  EPI == 2: weighted combine into out.
// EPI == 3: dense product, out[token][feature] = D (FP32, stride Hd).
// EPI == 4: SwiGLU -> FP32 H -> q8_1 of each 32-feature block (the integer
// route's first product; Hq, Hds, and H itself when Hf is given).
// WF: the weight format, IQ4_NL (raw stages of 4 k-steps) or Q8_0 (2).
// PAIR: CTA pairs (clusters of two) on neighbouring feature tiles of the same
// token tile share M = 256 MMAs (tcgen05 cta_group::2): each CTA dequantises
// its own 128 weight rows into its own TMEM and loads its own half of the
// token rows with TMA (no multicast), so every SM writes and the MMA reads
// half of the tile's token bytes per k-step; both CTAs' loads count their
// bytes on the even CTA's stage barrier (cta_group::2 loads), and the even
// CTA issues the MMAs and commits them to the barriers of both CTAs.  A pair's tile has up to
// 384 tokens in two sub-tiles (two accumulator slots), so each dequantised
// weight stage feeds twice the MMA work of a 192-token tile.  !PAIR: one CTA,
// M = 128, tiles of up to 192 tokens.
template <int EPI, bool PAIR, int WF>
__global__ void __launch_bounds__(PF_THREADS, 1) prefill_gemm_kernel(const __grid_constant__ CUtensorMap bmap,
                                                                     const __grid_constant__ CUtensorMap qmap,
                                                                     const __grid_constant__ CUtensorMap smap,
                                                                     GemmArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const PfSmem L;
  constexpr int HALF_B = pf_rows_cta<EPI, PAIR>() * PF_BOXK * 2;  // bytes of one 64-input half of a B stage
  constexpr int STAGE_B = 2 * HALF_B;                              // bytes of one B stage
  constexpr int NB = PF_B_BYTES / STAGE_B;                         // B stages
  static_assert(NB <= PF_NB_MAX && PF_KD % NB == 0, "B stages free on the k-step-done ring");
  uint8_t* sb = smem + L.b;
  uint8_t* sraw = smem + L.raw;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L.bars);
  // k-step kc uses B stage kc % NB and A stage kc % PF_NA_ST; its one
  // MMA commit (for a pair, to both CTAs) completes kdone[kc % PF_KD], which
  // frees both stages
  // b_full[s]: the B stage has landed (for a pair, on the issuing CTA: both
  // CTAs' halves, whose loads both count their bytes on it)
  uint64_t* b_full = bars;
  uint64_t* kdone = b_full + NB;
  // full[s] (on the CTA that issues the MMAs): the A stage is in TMEM in
  // every CTA of the pair (each dequantising warp arrives; the odd CTA's
  // remotely)
  uint64_t* full = kdone + PF_KD;
  uint64_t* d_full = full + PF_NA_ST;       // accumulator slot h holds a finished sub-tile
  uint64_t* d_empty = d_full + 2;           // accumulator slot h has been read by every epilogue warp
  uint64_t* done_bar = d_empty + 2;
  uint64_t* r_full = done_bar + 1;
  uint64_t* r_empty = r_full + PF_NR_ST;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + L.tmem);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L.abort_flag);
  constexpr int BOXR = pf_boxr<PAIR>();
  constexpr bool GU = EPI == 1 || EPI == 4;  // GEMM 1: gate and up rows of 64 features
  float* xch = reinterpret_cast<float*>(smem + L.xch);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < NB; ++i) mbar_init(&b_full[i], 1);
    for (int i = 0; i < PF_KD; ++i) mbar_init(&kdone[i], 1);  // the MMA thread's commit
    for (int i = 0; i < PF_NA_ST; ++i) mbar_init(&full[i], PAIR ? 2 * PF_DQ_WARPS : PF_DQ_WARPS);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&d_full[i], 1);
      mbar_init(&d_empty[i], (PAIR ? 2 : 1) * PF_EPI_WARPS);  // every epilogue warp (of both CTAs of a pair)
    }
    mbar_init(done_bar, 1);
    for (int i = 0; i < PF_NR_ST; ++i) {
      mbar_init(&r_full[i], 1);
      mbar_init(&r_empty[i], PF_DQ_WARPS);
    }
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&bmap);
    tma_prefetch_desc(&qmap);
    tma_prefetch_desc(&smap);
  }
  if (warp == 1) {
    if constexpr (PAIR) {
      tmem_alloc_pair(tmem_holder, 512);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(tmem_holder, 512);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  __syncthreads();
  if (PAIR) cluster_sync_all();  // both CTAs' barriers are initialised before any remote arrival
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;

  pdl_wait();  // tiles, tokens and (GEMM 2) H come from earlier kernels
  pdl_launch_dependents();
  // tiles 2p and 2p+1 (same expert and tokens, neighbouring feature tiles)
  // go to the two CTAs of one pair
  const int rank = PAIR ? static_cast<int>(cluster_ctarank()) : 0;
  const int t0 = PAIR ? 2 * (blockIdx.x >> 1) + rank : blockIdx.x;
  const int tstep = PAIR ? 2 * (gridDim.x >> 1) : gridDim.x;
  const int ntiles = *a.ntiles;
  const int KS = (a.K + PF_BK - 1) / PF_BK;   // k-steps; the last takes one half when K % 128 == 64
  const bool half_last = (a.K % PF_BK) != 0;

  if (warp == 0) {
    // ------------------------------------------------ B producer (TMA of this CTA's token rows)
    if (lane == 0) {
      const uint32_t b_full_mma = PAIR ? cluster_addr(smem_u32(b_full), 0) : 0u;
      int kc = 0;
      int4 nxt = t0 < ntiles ? a.tiles[t0] : make_int4(0, 0, 0, 0);
      for (int t = t0; t < ntiles && !*abort_flag; t += tstep) {
        const int4 tile = nxt;
        if (t + tstep < ntiles) nxt = a.tiles[t + tstep];  // read one tile ahead
        const PfSubTiles<PAIR> st(tile.w);
        int src[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) src[h] = tile.z + st.start[h] + (PAIR ? rank * (st.n[h] / 2) : 0);
        const uint32_t half_bytes = (st.nbox[0] + st.nbox[1]) * BOXR * PF_BOXK * 2;  // one CTA's
        for (int ks = 0; ks < KS; ++ks, ++kc) {
          const int s = kc % NB;
          const int j0 = kc - NB;  // the k-step that used this stage before
          if (j0 >= 0 && !mbar_wait(&kdone[j0 % PF_KD], (j0 / PF_KD) & 1, abort_flag)) {
            *abort_flag = 1;
            flag_status(a.status, DEV_TIMEOUT_MMA);
            break;
          }
          const int nhalf = (half_last && ks == KS - 1) ? 1 : 2;
          // a pair's two CTAs load the same number of boxes
          if (rank == 0) mbar_arrive_expect_tx(&b_full[s], (PAIR ? 2 : 1) * nhalf * half_bytes);
          for (int j = 0; j < nhalf; ++j)
#pragma unroll
            for (int h = 0; h < 2; ++h)
              for (int bx = 0; bx < st.nbox[h]; ++bx) {
                uint8_t* dst = sb + s * STAGE_B + j * HALF_B + (st.off[h] + bx * BOXR) * PF_BOXK * 2;
                if constexpr (PAIR)
                  tma_load_2d_pair(dst, &bmap, ks * PF_BK + j * PF_BOXK, src[h] + BOXR * bx, b_full_mma + 8u * s);
                else
                  tma_load_2d(dst, &bmap, ks * PF_BK + j * PF_BOXK, src[h] + BOXR * bx, &b_full[s]);
              }
        }
      }
      // after an abort, let the copies already issued land before the CTA
      // exits: the issuing CTA waits for its stages (which count the odd
      // CTA's bytes too); the odd CTA, which cannot wait on that barrier,
      // gives its copies a fixed 100 us
      if (*abort_flag) {
        if (rank == 0) {
          for (int j = kc - 1; j >= 0 && j >= kc - NB; --j)
            mbar_wait(&b_full[j % NB], (j / NB) & 1, nullptr);
        } else {
          const uint64_t t_ab = global_timer_ns();
          while (global_timer_ns() - t_ab < 100000ull) __nanosleep(1000);
        }
      }
    }
  } else if (warp == 1 && PAIR && rank == 1) {
    // the odd CTA of a pair issues no MMAs
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer (one CTA, or the even CTA of a pair)
    if (lane == 0) {
      uint32_t kdone_peer = 0, d_full_peer = 0;
      if constexpr (PAIR) {
        kdone_peer = cluster_addr(smem_u32(kdone), 1);
        d_full_peer = cluster_addr(smem_u32(d_full), 1);
      }
      int kc = 0;
      int nsub = 0;  // sub-tiles so far: sub-tile number i accumulates in slot i & 1 (its use i >> 1)
      bool issued_any = false;
      int4 nxt = t0 < ntiles ? a.tiles[t0] : make_int4(0, 0, 0, 0);
      for (int t = t0; t < ntiles && !*abort_flag; t += tstep) {
        const int4 tile = nxt;
        if (t + tstep < ntiles) nxt = a.tiles[t + tstep];
        const PfSubTiles<PAIR> st(tile.w);
        // everything the k-loop needs, computed once a tile: per sub-tile the
        // instruction descriptor, the D column and the B descriptor of stage 0
        // (a stage or a 16-input step only adds to its 14-bit address field)
        const int nh = st.n[1] > 0 ? 2 : 1;
        uint32_t idesc[2], dcol[2];
        uint64_t bdesc[2];
        int sub[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          sub[h] = nsub + h;
          idesc[h] = idesc_f16_f32(PAIR ? 256 : 128, st.n[h] > 0 ? st.n[h] : 16);
          dcol[h] = tmem + (sub[h] & 1) * PF_SUBN;
          bdesc[h] = smem_desc_sw128(smem_u32(sb) + st.off[h] * PF_BOXK * 2);
        }
        // the slots' previous sub-tiles must have been read out first
        bool ok = true;
        for (int h = 0; h < nh && ok; ++h)
          if (sub[h] >= 2) ok = mbar_wait(&d_empty[sub[h] & 1], ((sub[h] >> 1) - 1) & 1, abort_flag);
        if (!ok) {
          *abort_flag = 1;
          flag_status(a.status, DEV_TIMEOUT_MMA);
          break;
        }
        for (int ks = 0; ks < KS; ++ks, ++kc) {
          const int sb_ = kc % NB, sa = kc % PF_NA_ST;
          if (!mbar_wait(&b_full[sb_], (kc / NB) & 1, abort_flag) ||
              !mbar_wait(&full[sa], (kc / PF_NA_ST) & 1, abort_flag)) {
            *abort_flag = 1;
            flag_status(a.status, DEV_TIMEOUT_MMA);
            break;
          }
          tc_fence_after();
          const uint32_t acol = tmem + PF_ACOL + sa * PF_ACOLS;
          const uint64_t boff = static_cast<uint64_t>((sb_ * STAGE_B) >> 4);
          const int nkk = (half_last && ks == KS - 1) ? PF_BOXK / 16 : PF_BK / 16;
          for (int h = 0; h < nh; ++h) {
            for (int kk = 0; kk < nkk; ++kk) {
              // 16-input step kk: half kk / 4 of the stage, 32 bytes further per step within it
              const uint64_t bd = bdesc[h] + boff + (kk >> 2) * (HALF_B >> 4) + 2 * (kk & 3);
              if constexpr (PAIR)
                mma_f16_ts_pair(dcol[h], acol + kk * 8, bd, idesc[h], (ks | kk) != 0);
              else
                mma_f16_ts(dcol[h], acol + kk * 8, bd, idesc[h], (ks | kk) != 0);
            }
          }
          issued_any = true;
          if constexpr (PAIR) {
            mma_commit_pair(smem_u32(&kdone[kc % PF_KD]));
            mma_commit_pair(kdone_peer + 8u * (kc % PF_KD));
          } else {
            mma_commit(&kdone[kc % PF_KD]);
          }
        }
        if (*abort_flag) break;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          if (st.n[h] == 0) continue;
          const int sl = sub[h] & 1;
          if constexpr (PAIR) {
            mma_commit_pair(smem_u32(&d_full[sl]));
            mma_commit_pair(d_full_peer + 8u * sl);
          } else {
            mma_commit(&d_full[sl]);
          }
          ++nsub;
        }
      }
      // make sure no MMA is still running before the TMEM is released
      if (issued_any) {
        if constexpr (PAIR)
          mma_commit_pair(smem_u32(done_bar));
        else
          mma_commit(done_bar);
        mbar_wait(done_bar, 0, nullptr);
      }
    }
  } else if (warp == 2) {
    // ------------------------------------------------ A producer (TMA of the raw weight bytes)
    if (lane == 0) {
      int rc = 0;
      constexpr int RKS = pf_raw_ks(WF);
      const int ngroups = (KS + RKS - 1) / RKS;
      int4 nxt = t0 < ntiles ? a.tiles[t0] : make_int4(0, 0, 0, 0);
      for (int t = t0; t < ntiles && !*abort_flag; t += tstep) {
        const int4 tile = nxt;
        if (t + tstep < ntiles) nxt = a.tiles[t + tstep];  // read one tile ahead
        const int64_t base = static_cast<int64_t>(tile.x) * a.rows_per_expert;
        // weight rows of raw rows 0..63 and 64..127: gate and up features (GEMM 1) or 128 outputs (GEMM 2)
        const int y0 = static_cast<int>(GU ? base + tile.y * 64 : base + tile.y * 128);
        const int y1 = static_cast<int>(GU ? base + a.I + tile.y * 64 : base + tile.y * 128 + 64);
        for (int g = 0; g < ngroups; ++g, ++rc) {
          const int r = rc % PF_NR_ST;
          if (rc >= PF_NR_ST && !mbar_wait(&r_empty[r], ((rc / PF_NR_ST) - 1) & 1, abort_flag)) {
            *abort_flag = 1;
            flag_status(a.status, DEV_TIMEOUT_PIPE);
            break;
          }
          uint8_t* st = sraw + r * PF_RAW_STAGE;
          mbar_arrive_expect_tx(&r_full[r], PF_RAW_STAGE);
          tma_load_2d(st, &qmap, g * 128, y0, &r_full[r]);
          tma_load_2d(st + 64 * 128, &qmap, g * 128, y1, &r_full[r]);
          // scales: 16 bytes = 4 k-steps (a Q8_0 stage of 2 k-steps takes half of it)
          const int sx = (WF == MOEX_Q8_0 ? g >> 1 : g) * 16;
          tma_load_2d(st + PF_RAW_QS, &smap, sx, y0, &r_full[r]);
          tma_load_2d(st + PF_RAW_QS + 64 * 16, &smap, sx, y1, &r_full[r]);
        }
      }
      if (*abort_flag) {
        for (int j = rc - 1; j >= 0 && j >= rc - PF_NR_ST; --j)
          mbar_wait(&r_full[j % PF_NR_ST], (j / PF_NR_ST) & 1, nullptr);
      }
    }
  } else if (warp < PF_EPI0) {
    // ------------------------------------------------ dequantise into TMEM
    // warp pair (w, w + 4) shares lane quarter q; half h dequantises blocks
    // 2h and 2h + 1 of each 128-input k-step (TMEM columns 32h .. 32h+31 of
    // the stage).
    const int q = warp & 3;
    const int h = (warp - PF_DQ0) >> 2;
    const int m = 32 * q + lane;                          // A row = TMEM lane
    const int rr = GU ? pf_gu_raw_row(m) : m;             // its row in the raw stage
    // raw stage rows: 128 bytes, 16-byte chunk c stored at chunk c ^ (row & 7)
    const int qoff = (rr >> 6) * 64 * 128 + (rr & 63) * 128;
    const int soff = PF_RAW_QS + (rr >> 6) * 64 * 16 + (rr & 63) * 16;
    constexpr int RKS = pf_raw_ks(WF);
    const int ngroups = (KS + RKS - 1) / RKS;
    const uint32_t full_mma = PAIR ? cluster_addr(smem_u32(full), 0) : 0;  // the issuing CTA's full barriers
    int kc = 0, rc = 0;
    for (int t = t0; t < ntiles && !*abort_flag; t += tstep) {
      for (int g = 0; g < ngroups && !*abort_flag; ++g, ++rc) {
        const int r = rc % PF_NR_ST;
        if (!mbar_wait(&r_full[r], (rc / PF_NR_ST) & 1, abort_flag)) {
          *abort_flag = 1;
          flag_status(a.status, DEV_TIMEOUT_PIPE);
          break;
        }
        const uint8_t* st = sraw + r * PF_RAW_STAGE;
        const int nk = min(RKS, KS - g * RKS);
        const uint4 scv = *reinterpret_cast<const uint4*>(st + soff);
        // block b = 2h + i of the stage's k-step j: IQ4_NL 16 bytes (chunk 4j + b),
        // Q8_0 32 bytes (chunks 2b, 2b + 1; one k-step a stage)
        constexpr int NCH = WF == MOEX_Q8_0 ? 2 : 1;
        uint4 qv[RKS][2][NCH];
#pragma unroll
        for (int j = 0; j < RKS; ++j)
#pragma unroll
          for (int i = 0; i < 2; ++i)
#pragma unroll
            for (int c = 0; c < NCH; ++c)
              if (j < nk) {
                const int chunk = WF == MOEX_Q8_0 ? 2 * (2 * h + i) + c : 4 * j + 2 * h + i;
                qv[j][i][c] = *reinterpret_cast<const uint4*>(st + qoff + ((chunk ^ (rr & 7)) << 4));
              }
        __syncwarp();
        if (lane == 0) mbar_arrive(&r_empty[r]);  // the raw bytes are in registers
        const uint32_t sw[4] = {scv.x, scv.y, scv.z, scv.w};
#pragma unroll
        for (int j = 0; j < RKS; ++j) {
          if (j >= nk) break;
          const int ks = g * RKS + j;
          // a half last k-step has blocks 0 and 1 only
          const bool has = !(half_last && ks == KS - 1 && h == 1);
          const int sa = kc % PF_NA_ST;
          const int j0 = kc - PF_NA_ST;  // the k-step that used this A stage before
          if (j0 >= 0 && !mbar_wait(&kdone[j0 % PF_KD], (j0 / PF_KD) & 1, abort_flag)) {
            *abort_flag = 1;
            flag_status(a.status, DEV_TIMEOUT_MMA);
            break;
          }
          tc_fence_after();
          if (has) {
#pragma unroll
            for (int i = 0; i < 2; ++i) {
              // scale of block b = 2h + i: word 2j + h (Q8_0: 2 (g & 1) + h) of the 8 scales, half i
              const uint32_t swv = sw[WF == MOEX_Q8_0 ? 2 * (g & 1) + h : 2 * j + h];
              const uint16_t dbits = static_cast<uint16_t>(i ? (swv >> 16) : (swv & 0xFFFFu));
              uint32_t col[16];
              if constexpr (WF == MOEX_Q8_0)
                dequant_q8_block16(qv[j][i][0], qv[j][i][NCH - 1], dbits, col);
              else
                dequant_block16(qv[j][i][0], dbits, col);
              tmem_st16(tmem + (static_cast<uint32_t>(32 * q) << 16) + PF_ACOL + sa * PF_ACOLS + 32 * h + 16 * i, col);
            }
            tmem_st_wait();
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) {  // the warp's 32 rows of these blocks are in TMEM
            if (PAIR && rank == 1)
              mbar_arrive_remote(full_mma + 8u * sa);
            else
              mbar_arrive(&full[sa]);
          }
          ++kc;
        }
      }
    }
  } else {
    // ------------------------------------------------ epilogue
    // warp (q, half): TMEM lane quarter q, 32-column chunks c with c % 2 == half
    const int q = warp & 3;
    const int half = (warp - PF_EPI0) >> 2;
    // the accumulator is released to the MMA thread's CTA (the even CTA of a pair)
    const uint32_t d_empty_mma = PAIR ? cluster_addr(smem_u32(d_empty), 0) : smem_u32(d_empty);
    int nsub = 0;  // as the MMA thread: sub-tile number i is in slot i & 1
    // (GEMM 1) this CTA's slice of the output to initialise, spread over its
    // tiles so that the writes stay a small share of the DRAM time, with
    // streaming (evict-first) stores that leave the weights and token rows
    // in L2
    const int ethr = threadIdx.x - 32 * PF_EPI0;
    int64_t zcur = a.init_vec4 * blockIdx.x / gridDim.x;
    const int64_t zend = a.init_vec4 * (blockIdx.x + 1) / gridDim.x;
    const int mytiles = t0 < ntiles ? (ntiles - t0 + tstep - 1) / tstep : 0;
    const int64_t zchunk = (zend - zcur + mytiles - 1) / (mytiles > 0 ? mytiles : 1);
    auto init_out_to = [&](int64_t zlim) {
      if constexpr (EPI == 1) {
        for (int64_t z = zcur + ethr; z < zlim; z += 32 * PF_EPI_WARPS)
          __stcs(a.init_out + z, a.init_res ? __ldcs(a.init_res + z) : make_float4(0.f, 0.f, 0.f, 0.f));
        zcur = zlim;
      }
    };
    int4 nxt = t0 < ntiles ? a.tiles[t0] : make_int4(0, 0, 0, 0);
    for (int t = t0; t < ntiles && !*abort_flag; t += tstep) {
      const int4 tile = nxt;
      if (t + tstep < ntiles) nxt = a.tiles[t + tstep];
      const PfSubTiles<PAIR> st(tile.w);
      for (int hs = 0; hs < 2 && !*abort_flag; ++hs) {
        if (st.n[hs] == 0) continue;
        const int sl = nsub & 1;
        bool stop = !mbar_wait(&d_full[sl], (nsub >> 1) & 1, abort_flag);
        if (stop) {
          *abort_flag = 1;
          flag_status(a.status, DEV_TIMEOUT_MMA);
        }
        // (integer route) the two warps of a feature block exchange through
        // shared memory: both take the same decision before the hand-offs
        if constexpr (EPI == 4) stop = named_bar_or(2 + (q >> 1) + 2 * half, 64, stop);
        if (stop) break;
        ++nsub;
        tc_fence_after();
        const uint32_t dbase = tmem + (static_cast<uint32_t>(32 * q) << 16) + sl * PF_SUBN;
        const int row0 = tile.z + st.start[hs];   // sorted row of the slot's column 0
        const int nrows = st.rows[hs];
        const int nchunk = (nrows + 31) / 32;
        for (int c = half; c < nchunk; c += 2) {
          uint32_t r[32];
          tmem_ld32(dbase + 32 * c, r);
          tmem_ld_wait();
          if constexpr (EPI == 1) {
            // lane l: gate (bit 3 clear) or up row of feature f; partners l ^ 8 (up / gate of f) and
            // l ^ 16 (feature f +- 16); a gate lane finishes even columns, an up lane odd ones
            const bool up = (lane >> 3) & 1;
            const int F = tile.y * 64 + pf_gu_feature(32 * q + lane);     // intermediate index
            const int hcol = (F & ~31) + 2 * (F & 15);                      // H position of F (lanes < 16) and F + 16
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const uint32_t send = up ? r[2 * i] : r[2 * i + 1];
              const float other = __uint_as_float(__shfl_xor_sync(0xffffffffu, send, 8));
              const float g = up ? other : __uint_as_float(r[2 * i]);
              const float u = up ? __uint_as_float(r[2 * i + 1]) : other;
              const float hv = __fmul_rn(__fdividef(g, 1.0f + __expf(-g)), u);
              const uint32_t hb = __half_as_ushort(__float2half_rn(hv));
              const uint32_t hp = __shfl_xor_sync(0xffffffffu, hb, 16);
              const int p = 32 * c + 2 * i + (up ? 1 : 0);   // column of this lane's h
              if (lane < 16 && p < nrows)
                *reinterpret_cast<uint32_t*>(a.Hs + static_cast<int64_t>(row0 + p) * a.I + hcol) = hb | (hp << 16);
            }
          } else if constexpr (EPI == 4) {
            // as EPI 1 (lane l: gate or up row of feature F, a gate lane finishing
            // the even columns, an up lane the odd ones); a q8_1 block of H is the
            // 32 features of warps q and q ^ 1: amax and the sum of the quants are
            // reduced over the 16 lanes of a column in each warp, then exchanged
            const bool up = (lane >> 3) & 1;
            const int F = tile.y * 64 + pf_gu_feature(32 * q + lane);     // intermediate index
            const int bar_id = 2 + (q >> 1) + 2 * half;
            float* mine = xch + ((q >> 1) + 2 * half) * 128 + (q & 1) * 32;   // [amax | sums] x 32 columns
            const float* theirs = xch + ((q >> 1) + 2 * half) * 128 + ((q & 1) ^ 1) * 32;
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {   // columns 16 hf .. 16 hf + 15 (pairs i = 8 hf .. 8 hf + 7)
              float hv[8], mx[8];
#pragma unroll
              for (int ii = 0; ii < 8; ++ii) {
                const int i = 8 * hf + ii;
                const uint32_t send = up ? r[2 * i] : r[2 * i + 1];
                const float other = __uint_as_float(__shfl_xor_sync(0xffffffffu, send, 8));
                const float g = up ? other : __uint_as_float(r[2 * i]);
                const float u = up ? __uint_as_float(r[2 * i + 1]) : other;
                hv[ii] = __fmul_rn(__fdividef(g, 1.0f + __expf(-g)), u);
                float m_ = fabsf(hv[ii]);
                m_ = fmaxf(m_, __shfl_xor_sync(0xffffffffu, m_, 1));
                m_ = fmaxf(m_, __shfl_xor_sync(0xffffffffu, m_, 2));
                m_ = fmaxf(m_, __shfl_xor_sync(0xffffffffu, m_, 4));
                mx[ii] = fmaxf(m_, __shfl_xor_sync(0xffffffffu, m_, 16));
              }
              if ((lane & 0x17) == 0)
#pragma unroll
                for (int ii = 0; ii < 8; ++ii) mine[2 * (8 * hf + ii) + (up ? 1 : 0)] = mx[ii];
              named_bar_sync(bar_id, 64);
              int qv[8], sm[8];
              float dv[8];
#pragma unroll
              for (int ii = 0; ii < 8; ++ii) {
                const float amax = fmaxf(mx[ii], theirs[2 * (8 * hf + ii) + (up ? 1 : 0)]);
                dv[ii] = amax > 0.f ? __fdiv_rn(amax, 127.0f) : 0.f;
                qv[ii] = amax > 0.f ? static_cast<int>(roundf(__fdiv_rn(hv[ii], dv[ii]))) : 0;
                int s_ = qv[ii];
                s_ += __shfl_xor_sync(0xffffffffu, s_, 1);
                s_ += __shfl_xor_sync(0xffffffffu, s_, 2);
                s_ += __shfl_xor_sync(0xffffffffu, s_, 4);
                sm[ii] = s_ + __shfl_xor_sync(0xffffffffu, s_, 16);
              }
              if ((lane & 0x17) == 0)
#pragma unroll
                for (int ii = 0; ii < 8; ++ii) mine[64 + 2 * (8 * hf + ii) + (up ? 1 : 0)] = __int_as_float(sm[ii]);
              named_bar_sync(bar_id, 64);
#pragma unroll
              for (int ii = 0; ii < 8; ++ii) {
                const int col = 2 * (8 * hf + ii) + (up ? 1 : 0);
                const int p = 32 * c + col;   // column of this lane's h
                if (p < nrows) {
                  const int64_t row = row0 + p;
                  a.Hq[row * a.I + F] = static_cast<int8_t>(qv[ii]);
                  if (a.Hf) a.Hf[row * a.I + F] = hv[ii];
                  if ((q & 1) == 0 && (lane & 0x17) == 0) {
                    const int total = sm[ii] + __float_as_int(theirs[64 + col]);
                    a.Hds[row * (a.I / QK) + (F >> 5)] = make_float2(dv[ii], __fmul_rn(dv[ii], static_cast<float>(total)));
                  }
                }
              }
            }
          } else if constexpr (EPI == 3) {
            const int fo = tile.y * 128 + 32 * q + lane;   // output feature
            for (int i = 0; i < 32; ++i)
              if (32 * c + i < nrows) a.out[static_cast<int64_t>(row0 + 32 * c + i) * a.Hd + fo] = __uint_as_float(r[i]);
          } else {
            const int fo = tile.y * 128 + 32 * q + lane;   // output feature
            const int pl = 32 * c + lane;
            const int2 tw = pl < nrows ? a.tokw[row0 + pl] : make_int2(0, 0);
            for (int i = 0; i < 32; ++i) {
              const int tok = __shfl_sync(0xffffffffu, tw.x, i);
              const float wt = __int_as_float(__shfl_sync(0xffffffffu, tw.y, i));
              if (32 * c + i < nrows) red_add_f32(a.out + static_cast<int64_t>(tok) * a.Hd + fo, wt * __uint_as_float(r[i]));
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if (PAIR)
            mbar_arrive_remote(d_empty_mma + 8u * sl);
          else
            mbar_arrive(&d_empty[sl]);
        }
      }
      init_out_to(zcur + zchunk < zend ? zcur + zchunk : zend);
    }
    init_out_to(zend);  // a CTA without tiles (or one that stopped early)
  }
  tc_fence_before();
  __syncthreads();
  if (PAIR) cluster_sync_all();  // the pair's MMAs, commits and remote arrivals are all done
  if (warp == 1) {
    tc_fence_after();
    if constexpr (PAIR)
      tmem_dealloc_pair(tmem, 512);
    else
      tmem_dealloc(tmem, 512);
  }
}

// ----------------------------------------------------------------- integer route: down product

// The down product of the integer route (#1525 Change: q8_1 rows of H for the
// down product, the integer "MMQ" route): for a tile of 128 output features
// of one expert and up to 64 of its sorted rows,
//   o[f][p] = sum_b fp32(dw[f,b]) * d_h[p,b] * I[f,p,b],
//   I = sum_{i<32} qw[f,32b+i] * qh[p,32b+i]       (int32, dp4a chains)
// summed over the blocks b in order, then out[token(p)] += w * o (atomic).
// Each weight block is decoded once per tile into shared memory (IQ4_NL to
// the int8 byte order of iq4nl_lookup4, with H's words permuted to match)
// and applied to the tile's 64 rows; the next block's bytes are loaded into
// registers while the current one is multiplied.
constexpr int QD_ROWS = 128;     // output features per tile
constexpr int QD_TOK = 64;       // sorted rows per tile
constexpr int QD_THREADS = 256;  // warp w: rows 8w .. 8w+7, lane l: features l + 32j

struct Q8DownArgs {
  const uint8_t* qs;
  const uint8_t* sc;
  int qrow, scrow;
  int64_t rows_per_expert;
  int I;                 // inputs of the down product (multiple of 32)
  const int4* tiles;     // {expert, feature tile, first sorted row, rows}
  const int* ntiles;
  const int8_t* hq;      // [rows][I]
  const float2* hds;     // [rows][I/32] {d, s}
  const int2* tokw;      // per sorted row: token, weight bits
  float* out;            // [T][Hd], accumulated
  int Hd;
};

// Tile list of the integer down product: thread i of one 1024-thread CTA
// owns experts 4i .. 4i+3; each expert's rows are cut into balanced token
// tiles of at most 64 rows, each paired with every feature tile.
__global__ void __launch_bounds__(1024) q8_tiles_kernel(int E, int F, const int* __restrict__ counts,
                                                        const int* __restrict__ eoff, int4* __restrict__ tiles,
                                                        int* __restrict__ ntiles) {
  __shared__ int red[32];
  pdl_wait();
  pdl_launch_dependents();
  int nt[4];
  int sum = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int e = 4 * threadIdx.x + i;
    nt[i] = e < E ? pf_token_tiles(counts[e], QD_TOK) : 0;
    sum += nt[i];
  }
  int base = sum;
  const int total = block_exscan(base, red);
  if (threadIdx.x == 0) *ntiles = total * F;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int e = 4 * threadIdx.x + i;
    for (int tt = 0; tt < nt[i]; ++tt) {
      int r0, rows;
      pf_tile_span(counts[e], QD_TOK, tt, &r0, &rows);
      for (int f = 0; f < F; ++f) tiles[static_cast<int64_t>(base + tt) * F + f] = make_int4(e, f, eoff[e] + r0, rows);
    }
    base += nt[i];
  }
}

__device__ __forceinline__ uint4 ldg_nc16(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}

template <int FMT>
__global__ void __launch_bounds__(QD_THREADS) q8_down_kernel(Q8DownArgs a) {
  // decoded weight words of 128 rows (the two 16-byte halves of row r swapped
  // when bit 2 of r is set, so a quarter warp's 16-byte reads of 8 rows hit
  // 32 distinct banks) and H's words of 64 rows, double-buffered by block
  __shared__ __align__(16) uint32_t wsm[2][QD_ROWS * 8];
  __shared__ float wdm[2][QD_ROWS];
  __shared__ __align__(16) uint32_t xsm[2][QD_TOK * 8];
  __shared__ float xdm[2][QD_TOK];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  pdl_wait();
  pdl_launch_dependents();
  const int ntiles = *a.ntiles;
  const int NB = a.I / QK;
  for (int t = blockIdx.x; t < ntiles; t += gridDim.x) {
    const int4 tile = a.tiles[t];
    const int64_t wrow0 = static_cast<int64_t>(tile.x) * a.rows_per_expert + static_cast<int64_t>(tile.y) * QD_ROWS;
    // loaders: thread f < 128 fetches weight row f, thread 128 + p fetches H row p
    uint4 q0 = make_uint4(0, 0, 0, 0), q1 = q0;
    uint32_t sw = 0;
    float xd = 0.f;
    auto fetch = [&](int b) {
      if (tid < QD_ROWS) {
        const uint8_t* src = a.qs + (wrow0 + tid) * a.qrow + b * FmtTraits<FMT>::QBYTES;
        q0 = ldg_nc16(src);
        if (FMT == MOEX_Q8_0) q1 = ldg_nc16(src + 16);
        sw = *reinterpret_cast<const uint16_t*>(a.sc + (wrow0 + tid) * a.scrow + 2 * b);
      } else if (tid < QD_ROWS + QD_TOK) {
        const int p = tid - QD_ROWS;
        if (p < tile.w) {
          const int8_t* src = a.hq + static_cast<int64_t>(tile.z + p) * a.I + b * QK;
          q0 = *reinterpret_cast<const uint4*>(src);
          q1 = *reinterpret_cast<const uint4*>(src + 16);
          xd = a.hds[static_cast<int64_t>(tile.z + p) * NB + b].x;
        } else {
          q0 = q1 = make_uint4(0, 0, 0, 0);
          xd = 0.f;
        }
      }
    };
    auto stage = [&](int buf) {
      if (tid < QD_ROWS) {
        uint32_t wv[8];
        if constexpr (FMT == MOEX_Q8_0) {
          wv[0] = q0.x; wv[1] = q0.y; wv[2] = q0.z; wv[3] = q0.w;
          wv[4] = q1.x; wv[5] = q1.y; wv[6] = q1.z; wv[7] = q1.w;
        } else {
          const uint32_t W[4] = {q0.x, q0.y, q0.z, q0.w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const uint32_t fl = W[i] ^ 0x88888888u;
            wv[2 * i] = iq4nl_lookup4(W[i], fl);
            wv[2 * i + 1] = iq4nl_lookup4(W[i] >> 16, fl >> 16);
          }
        }
        const int sx = (tid >> 2) & 1;
        uint4* dst = reinterpret_cast<uint4*>(&wsm[buf][tid * 8]);
        dst[sx] = make_uint4(wv[0], wv[1], wv[2], wv[3]);
        dst[sx ^ 1] = make_uint4(wv[4], wv[5], wv[6], wv[7]);
        wdm[buf][tid] = __half2float(__ushort_as_half(static_cast<uint16_t>(sw)));
      } else if (tid < QD_ROWS + QD_TOK) {
        const int p = tid - QD_ROWS;
        uint32_t xv[8];
        const uint32_t X[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
        if constexpr (FMT == MOEX_Q8_0) {
#pragma unroll
          for (int i = 0; i < 8; ++i) xv[i] = X[i];
        } else {
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            xv[2 * i] = prmt(X[i], X[i + 4], 0x5140);
            xv[2 * i + 1] = prmt(X[i], X[i + 4], 0x7362);
          }
        }
        uint4* dst = reinterpret_cast<uint4*>(&xsm[buf][p * 8]);
        dst[0] = make_uint4(xv[0], xv[1], xv[2], xv[3]);
        dst[1] = make_uint4(xv[4], xv[5], xv[6], xv[7]);
        xdm[buf][p] = xd;
      }
    };
    fetch(0);
    stage(0);
    __syncthreads();
    float acc[4][8];
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[j][i] = 0.f;
    for (int b = 0; b < NB; ++b) {
      const int buf = b & 1;
      if (b + 1 < NB) fetch(b + 1);
      uint32_t wv[4][8];
      float dw[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int r = lane + 32 * j;
        const int sx = (r >> 2) & 1;
        const uint4* src = reinterpret_cast<const uint4*>(&wsm[buf][r * 8]);
        const uint4 lo = src[sx], hi = src[sx ^ 1];
        wv[j][0] = lo.x; wv[j][1] = lo.y; wv[j][2] = lo.z; wv[j][3] = lo.w;
        wv[j][4] = hi.x; wv[j][5] = hi.y; wv[j][6] = hi.z; wv[j][7] = hi.w;
        dw[j] = wdm[buf][r];
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int p = 8 * warp + i;
        const uint4* src = reinterpret_cast<const uint4*>(&xsm[buf][p * 8]);
        const uint4 lo = src[0], hi = src[1];
        const uint32_t xv[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
        const float dx = xdm[buf][p];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          int I = 0;
#pragma unroll
          for (int z = 0; z < 8; ++z) I = dp4a(wv[j][z], xv[z], I);
          acc[j][i] = __fadd_rn(acc[j][i], __fmul_rn(__int2float_rn(I), __fmul_rn(dw[j], dx)));
        }
      }
      if (b + 1 < NB) stage(buf ^ 1);
      __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int p = 8 * warp + i;
      if (p < tile.w) {
        const int2 tw = a.tokw[tile.z + p];
        const float wt = __int_as_float(tw.y);
        float* dst = a.out + static_cast<int64_t>(tw.x) * a.Hd + tile.y * QD_ROWS + lane;
#pragma unroll
        for (int j = 0; j < 4; ++j) red_add_f32(dst + 32 * j, wt * acc[j][i]);
      }
    }
  }
}

// ----------------------------------------------------------------- host side

namespace {

// 2-D FP16 map over [rows][cols] (row pitch cols*2 bytes), box 64 inputs x
// boxr rows, 128-byte swizzle.
bool make_map(CUtensorMap* m, void* base, int64_t rows, int64_t cols, int boxr) {
  EncodeTiledFn fn = encode_tiled_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols * 2)};
  const cuuint32_t box[2] = {PF_BOXK, static_cast<cuuint32_t>(boxr)};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D byte map over a weight plane: [rows][pitch] with `used` bytes a row,
// box box_x bytes x 64 rows.
bool make_plane_map(CUtensorMap* m, const void* base, int64_t rows, int64_t used, int64_t pitch, int box_x,
                    CUtensorMapSwizzle swz) {
  EncodeTiledFn fn = encode_tiled_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(used), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(pitch)};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(box_x), 64};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Quant map (box 128 bytes: 4 IQ4_NL k-steps or 2 Q8_0 k-steps, 128-byte
// swizzle) and scale map (box 16 bytes = the 8 scales of 4 k-steps) of a
// weight stack.
bool make_weight_maps(CUtensorMap* qm, CUtensorMap* sm, const moex_qweight* w) {
  const int64_t rows = static_cast<int64_t>(w->n_mats) * w->rows;
  const int64_t qused = w->fmt == MOEX_Q8_0 ? w->K : w->K / 2;  // quant bytes of a row
  return make_plane_map(qm, w->qs, rows, qused, qs_row_bytes(w->fmt, w->K), 128, CU_TENSOR_MAP_SWIZZLE_128B) &&
         make_plane_map(sm, w->scales, rows, w->K / 16, sc_row_bytes(w->K), 16, CU_TENSOR_MAP_SWIZZLE_NONE);
}

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

using PfKernel = void (*)(CUtensorMap, CUtensorMap, CUtensorMap, GemmArgs);

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
  static int cached[8] = {};
  static PfKernel which[8] = {};
  int slot = 0;
  for (; slot < 8 && which[slot]; ++slot)
    if (which[slot] == kern) return cached[slot];
  cudaLaunchAttribute attr[2];
  cudaLaunchConfig_t cfg = pf_config(sm_count(), smem, nullptr, cl, attr);
  int nclusters = 0;
  if (cudaOccupancyMaxActiveClusters(&nclusters, kern, &cfg) != cudaSuccess || nclusters <= 0) {
    cudaGetLastError();
    nclusters = sm_count() / 2;
  }
  if (slot == 8) return 2 * nclusters;
  which[slot] = kern;
  cached[slot] = 2 * nclusters;
  return cached[slot];
}

// cl == 2: the CTA-pair kernel; cl == 1: single CTAs.
template <int EPI>
PfKernel pf_kernel(int cl, int fmt) {
  if (fmt == MOEX_Q8_0)
    return cl == 2 ? prefill_gemm_kernel<EPI, true, MOEX_Q8_0> : prefill_gemm_kernel<EPI, false, MOEX_Q8_0>;
  return cl == 2 ? prefill_gemm_kernel<EPI, true, MOEX_IQ4_NL> : prefill_gemm_kernel<EPI, false, MOEX_IQ4_NL>;
}

int pf_boxr_host(int cl) { return cl == 2 ? pf_boxr<true>() : pf_boxr<false>(); }

cudaError_t launch_pf_gemm(PfKernel kern, int cl, size_t smem, cudaStream_t s, const CUtensorMap& bmap,
                           const CUtensorMap& qmap, const CUtensorMap& smap, const GemmArgs& args) {
  cudaLaunchAttribute attr[2];
  cudaLaunchConfig_t cfg = pf_config(pf_grid(kern, cl, smem), smem, s, cl, attr);
  return cudaLaunchKernelEx(&cfg, kern, bmap, qmap, smap, args);
}

}  // namespace

// Workspace layout (offsets in bytes, each 256-aligned).
void prefill_ws_layout(int T, int k, int E, int64_t hidden, int64_t inter, size_t* off) {
  const size_t n = static_cast<size_t>(T) * k;
  const size_t tiles = n / PF_CAP_ONE + E + 1;   // token tiles of both tile caps fit
  const size_t segs = static_cast<size_t>(pf_nsegs(static_cast<int>(n)));
  size_t o = 0;
  off[0] = o; o = align_up(o + 4 * E + 4 * segs * E + 8 * E + 4 + 4 * n, 256);  // counts, segment histograms, eoff, etb, pos
  off[1] = o; o = align_up(o + 4 * n, 256);                              // order
  off[2] = o; o = align_up(o + 8 * n, 256);                              // tokw
  off[3] = o; o = align_up(o + 16 * tiles * (inter / 64), 256);          // tiles 1
  off[4] = o; o = align_up(o + 16 * tiles * (hidden / 128), 256);        // tiles 2
  off[5] = o; o = align_up(o + 16, 256);                                 // n1, n2, placed rows
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
                               const int32_t* ids, const float* w, int k, const float* residual, float* out, void* ws,
                               cudaStream_t s) {
  const int E = gu->n_mats;
  const int H = static_cast<int>(gu->K), I = static_cast<int>(dn->K);
  const int n = T * k;
  size_t off[9];
  prefill_ws_layout(T, k, E, H, I, off);
  uint8_t* wsb = static_cast<uint8_t*>(ws);
  int* counts = reinterpret_cast<int*>(wsb + off[0]);
  int* order = reinterpret_cast<int*>(wsb + off[1]);
  int2* tokw = reinterpret_cast<int2*>(wsb + off[2]);
  // CTA pairs share each MMA when both GEMMs have an even number of feature tiles
  const int cl = (I / 64) % 2 == 0 && (H / 128) % 2 == 0 ? 2 : 1;
  PrefillTiles tl;
  tl.t1 = reinterpret_cast<int4*>(wsb + off[3]);
  tl.t2 = reinterpret_cast<int4*>(wsb + off[4]);
  tl.n1 = reinterpret_cast<int*>(wsb + off[5]);
  tl.n2 = tl.n1 + 1;
  tl.F1 = I / 64;
  tl.F2 = H / 128;
  // token tiles of at most 192 rows: one accumulator slot each, so the two
  // slots double-buffer and the SwiGLU / combine epilogues of a tile run
  // under the next tile's MMAs
  tl.cap = PF_CAP_ONE;
  __half* xs = reinterpret_cast<__half*>(wsb + off[6]);
  __half* hs = reinterpret_cast<__half*>(wsb + off[7]);
  uint32_t* status = device_status_ptr();

  CUtensorMap m1, m2, q1, s1, q2, s2;
  if (!make_map(&m1, xs, n, H, pf_boxr_host(cl)) || !make_map(&m2, hs, n, I, pf_boxr_host(cl)) ||
      !make_weight_maps(&q1, &s1, gu) || !make_weight_maps(&q2, &s2, dn))
    return MOEX_ECUDA;

  int* hist = counts + E;
  const int S = pf_nsegs(n);
  const size_t esm = static_cast<size_t>(E) * sizeof(int);
  if (launch_pdl(prefill_hist_kernel, dim3(S), dim3(256), esm, s, ids, n, E, hist, status) != cudaSuccess)
    return MOEX_ECUDA;
  int* eoff = hist + static_cast<int64_t>(S) * E;
  int* etb = eoff + E;
  if (launch_pdl(prefill_scan_kernel, dim3(1), dim3(1024), 0, s, n, E, hist, counts, eoff, etb, tl) != cudaSuccess)
    return MOEX_ECUDA;
  const int64_t max_tiles = (static_cast<int64_t>(n) / PF_CAP_ONE + E + 1) * (tl.F1 + tl.F2);
  if (launch_pdl(prefill_tiles_kernel, dim3(static_cast<unsigned>((max_tiles + 255) / 256)), dim3(256), esm + 4, s, E,
                 static_cast<const int*>(counts), static_cast<const int*>(eoff), static_cast<const int*>(etb),
                 tl) != cudaSuccess)
    return MOEX_ECUDA;
  int* pos = etb + E + 1;  // each entry's sorted row
  if (launch_pdl(prefill_scatter_kernel, dim3(S), dim3(32), esm, s, ids, w, n, k, E, static_cast<const int*>(hist),
                 order, tokw, pos) != cudaSuccess)
    return MOEX_ECUDA;
  if (launch_pdl(prefill_gather_kernel, dim3(static_cast<unsigned>((T + 7) / 8)), dim3(256), 0, s, x, H, T, k,
                 static_cast<const int*>(pos), xs, static_cast<const float4*>(nullptr), static_cast<float4*>(nullptr),
                 int64_t(0)) != cudaSuccess)
    return MOEX_ECUDA;
  const PfSmem L;
  const PfKernel k1 = pf_kernel<1>(cl, gu->fmt);
  const PfKernel k2 = pf_kernel<2>(cl, dn->fmt);
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
  g1.init_out = reinterpret_cast<float4*>(out);
  g1.init_res = reinterpret_cast<const float4*>(residual);
  g1.init_vec4 = static_cast<int64_t>(T) * H / 4;
  g1.status = status;
  if (launch_pf_gemm(k1, cl, L.total, s, m1, q1, s1, g1) != cudaSuccess) return MOEX_ECUDA;
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
  if (launch_pf_gemm(k2, cl, L.total, s, m2, q2, s2, g2) != cudaSuccess) return MOEX_ECUDA;
  return MOEX_OK;
}

// Integer-route workspace: the sort (as the FP16 route), the GEMM 1 tile
// list, the down product's tile list (64-row token tiles), totals, Xs, and
// H as q8_1 rows (quants, then {d, s} per block).
void prefill_q8_ws_layout(int T, int k, int E, int64_t hidden, int64_t inter, size_t* off) {
  const size_t n = static_cast<size_t>(T) * k;
  const size_t segs = static_cast<size_t>(pf_nsegs(static_cast<int>(n)));
  size_t o = 0;
  off[0] = o; o = align_up(o + 4 * E + 4 * segs * E + 8 * E + 4 + 4 * n, 256);
  off[1] = o; o = align_up(o + 4 * n, 256);
  off[2] = o; o = align_up(o + 8 * n, 256);
  off[3] = o; o = align_up(o + 16 * (n / PF_CAP_ONE + E + 1) * (inter / 64), 256);
  off[4] = o; o = align_up(o + 16 * (n / QD_TOK + E + 1) * (hidden / QD_ROWS), 256);
  off[5] = o; o = align_up(o + 32, 256);                                  // totals (GEMM 1 ..., down tiles at [4])
  off[6] = o; o = align_up(o + 2 * n * hidden, 256);                      // Xs
  off[7] = o; o = align_up(o + n * inter, 256);                           // Hq
  off[8] = o; o = align_up(o + 8 * n * (inter / QK), 256);                // {d, s}
  off[9] = o;
}

size_t moe_prefill_q8_ws_bytes(int T, int k, int E, int64_t hidden, int64_t inter) {
  size_t off[10];
  prefill_q8_ws_layout(T, k, E, hidden, inter, off);
  return off[9];
}

moex_status launch_moe_prefill_q8(const moex_qweight* gu, const moex_qweight* dn, const uint16_t* x, int T,
                                  const int32_t* ids, const float* w, int k, float* out, void* ws, float* h_dbg,
                                  cudaStream_t s) {
  const int E = gu->n_mats;
  const int H = static_cast<int>(gu->K), I = static_cast<int>(dn->K);
  const int n = T * k;
  size_t off[10];
  prefill_q8_ws_layout(T, k, E, H, I, off);
  uint8_t* wsb = static_cast<uint8_t*>(ws);
  int* counts = reinterpret_cast<int*>(wsb + off[0]);
  int* order = reinterpret_cast<int*>(wsb + off[1]);
  int2* tokw = reinterpret_cast<int2*>(wsb + off[2]);
  const int cl = (I / 64) % 2 == 0 ? 2 : 1;
  PrefillTiles tl;
  tl.t1 = reinterpret_cast<int4*>(wsb + off[3]);
  tl.t2 = tl.t1;                     // no tcgen05 GEMM 2 in this route: its list is left empty
  tl.n1 = reinterpret_cast<int*>(wsb + off[5]);
  tl.n2 = tl.n1 + 1;
  tl.F1 = I / 64;
  tl.F2 = 0;
  tl.cap = PF_CAP_ONE;
  int4* qt = reinterpret_cast<int4*>(wsb + off[4]);
  int* nq = tl.n1 + 4;
  __half* xs = reinterpret_cast<__half*>(wsb + off[6]);
  int8_t* hq = reinterpret_cast<int8_t*>(wsb + off[7]);
  float2* hds = reinterpret_cast<float2*>(wsb + off[8]);
  uint32_t* status = device_status_ptr();

  CUtensorMap m1, q1, s1;
  if (!make_map(&m1, xs, n, H, pf_boxr_host(cl)) || !make_weight_maps(&q1, &s1, gu)) return MOEX_ECUDA;
  int* hist = counts + E;
  const int S = pf_nsegs(n);
  const size_t esm = static_cast<size_t>(E) * sizeof(int);
  if (launch_pdl(prefill_hist_kernel, dim3(S), dim3(256), esm, s, ids, n, E, hist, status) != cudaSuccess)
    return MOEX_ECUDA;
  int* eoff = hist + static_cast<int64_t>(S) * E;
  int* etb = eoff + E;
  if (launch_pdl(prefill_scan_kernel, dim3(1), dim3(1024), 0, s, n, E, hist, counts, eoff, etb, tl) != cudaSuccess)
    return MOEX_ECUDA;
  const int64_t max_tiles = (static_cast<int64_t>(n) / PF_CAP_ONE + E + 1) * tl.F1;
  if (launch_pdl(prefill_tiles_kernel, dim3(static_cast<unsigned>((max_tiles + 255) / 256)), dim3(256), esm + 4, s, E,
                 static_cast<const int*>(counts), static_cast<const int*>(eoff), static_cast<const int*>(etb),
                 tl) != cudaSuccess)
    return MOEX_ECUDA;
  if (launch_pdl(q8_tiles_kernel, dim3(1), dim3(1024), 0, s, E, H / QD_ROWS, static_cast<const int*>(counts),
                 static_cast<const int*>(eoff), qt, nq) != cudaSuccess)
    return MOEX_ECUDA;
  int* pos = etb + E + 1;  // each entry's sorted row
  if (launch_pdl(prefill_scatter_kernel, dim3(S), dim3(32), esm, s, ids, w, n, k, E, static_cast<const int*>(hist),
                 order, tokw, pos) != cudaSuccess)
    return MOEX_ECUDA;
  if (launch_pdl(prefill_gather_kernel, dim3(static_cast<unsigned>((T + 7) / 8)), dim3(256), 0, s, x, H, T, k,
                 static_cast<const int*>(pos), xs, static_cast<const float4*>(nullptr), reinterpret_cast<float4*>(out),
                 static_cast<int64_t>(T) * H / 4) != cudaSuccess)
    return MOEX_ECUDA;
  const PfSmem L;
  const PfKernel k1 = pf_kernel<4>(cl, gu->fmt);
  if (ensure_smem(reinterpret_cast<const void*>(k1), L.total) != cudaSuccess) return MOEX_ECUDA;
  GemmArgs g1 = {};
  g1.qs = static_cast<const uint8_t*>(gu->qs);
  g1.sc = static_cast<const uint8_t*>(gu->scales);
  g1.qrow = static_cast<int>(qs_row_bytes(gu->fmt, gu->K));
  g1.scrow = static_cast<int>(sc_row_bytes(gu->K));
  g1.rows_per_expert = gu->rows;
  g1.K = H;
  g1.tiles = tl.t1;
  g1.ntiles = tl.n1;
  g1.Hq = hq;
  g1.Hds = hds;
  g1.Hf = h_dbg;
  g1.I = I;
  g1.status = status;
  if (launch_pf_gemm(k1, cl, L.total, s, m1, q1, s1, g1) != cudaSuccess) return MOEX_ECUDA;
  Q8DownArgs d = {};
  d.qs = static_cast<const uint8_t*>(dn->qs);
  d.sc = static_cast<const uint8_t*>(dn->scales);
  d.qrow = static_cast<int>(qs_row_bytes(dn->fmt, dn->K));
  d.scrow = static_cast<int>(sc_row_bytes(dn->K));
  d.rows_per_expert = dn->rows;
  d.I = I;
  d.tiles = qt;
  d.ntiles = nq;
  d.hq = hq;
  d.hds = hds;
  d.tokw = tokw;
  d.out = out;
  d.Hd = H;
  auto kd = dn->fmt == MOEX_Q8_0 ? q8_down_kernel<MOEX_Q8_0> : q8_down_kernel<MOEX_IQ4_NL>;
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kd, QD_THREADS, 0) != cudaSuccess || per_sm < 1) per_sm = 1;
  return cuda_status(launch_pdl(kd, dim3(sm_count() * per_sm), dim3(QD_THREADS), 0, s, d));
}

// Dense prefill workspace: tiles, totals, Xs.
void dense_ws_layout(int T, int64_t rows, int64_t K, size_t* off) {
  const size_t tiles = static_cast<size_t>(pf_token_tiles(T, PF_CAP_ONE)) * static_cast<size_t>(rows / 128);
  size_t o = 0;
  off[0] = o; o = align_up(o + 16 * tiles, 256);                     // tiles
  off[1] = o; o = align_up(o + 16, 256);                             // totals
  off[2] = o; o = align_up(o + 2 * static_cast<size_t>(T) * K, 256); // Xs
  off[3] = o;
}

size_t dense_prefill_ws_bytes(int T, int64_t rows, int64_t K) {
  size_t off[4];
  dense_ws_layout(T, rows, K, off);
  return off[3];
}

moex_status launch_dense_prefill(const moex_qweight* W, const uint16_t* x, int T, float* y, int64_t ldy, void* ws,
                                 cudaStream_t s) {
  const int K = static_cast<int>(W->K);
  const int F = static_cast<int>(W->rows / 128);
  size_t off[4];
  dense_ws_layout(T, W->rows, K, off);
  uint8_t* wsb = static_cast<uint8_t*>(ws);
  int4* tiles = reinterpret_cast<int4*>(wsb + off[0]);
  int* n1 = reinterpret_cast<int*>(wsb + off[1]);
  __half* xs = reinterpret_cast<__half*>(wsb + off[2]);
  uint32_t* status = device_status_ptr();
  const int cl = F % 2 == 0 ? 2 : 1;
  CUtensorMap bm, qm, sm;
  if (!make_map(&bm, xs, T, K, pf_boxr_host(cl)) || !make_weight_maps(&qm, &sm, W)) return MOEX_ECUDA;
  // a pair takes tiles of up to 384 tokens (two accumulator slots): each
  // dequantised weight stage feeds twice the MMA work, and the plain-store
  // epilogue is short enough to leave exposed
  const int cap = cl == 2 ? PF_CAP_PAIR : PF_CAP_ONE;
  const int ntiles = pf_token_tiles(T, cap) * F;
  if (launch_pdl(dense_tiles_kernel, dim3((ntiles + 255) / 256), dim3(256), 0, s, T, F, cap, tiles, n1) != cudaSuccess)
    return MOEX_ECUDA;
  if (launch_pdl(prefill_gather_kernel, dim3(static_cast<unsigned>((T + 7) / 8)), dim3(256), 0, s, x, K, T, 1,
                 static_cast<const int*>(nullptr), xs, static_cast<const float4*>(nullptr), static_cast<float4*>(nullptr),
                 int64_t(0)) != cudaSuccess)
    return MOEX_ECUDA;
  const PfSmem L;
  const PfKernel kern = pf_kernel<3>(cl, W->fmt);
  if (ensure_smem(reinterpret_cast<const void*>(kern), L.total) != cudaSuccess) return MOEX_ECUDA;
  GemmArgs g = {};
  g.qs = static_cast<const uint8_t*>(W->qs);
  g.sc = static_cast<const uint8_t*>(W->scales);
  g.qrow = static_cast<int>(qs_row_bytes(W->fmt, W->K));
  g.scrow = static_cast<int>(sc_row_bytes(W->K));
  g.rows_per_expert = W->rows;
  g.K = K;
  g.tiles = tiles;
  g.ntiles = n1;
  g.out = y;
  g.Hd = static_cast<int>(ldy);
  g.status = status;
  if (launch_pf_gemm(kern, cl, L.total, s, bm, qm, sm, g) != cudaSuccess) return MOEX_ECUDA;
  return MOEX_OK;
}

}  // namespace moex
