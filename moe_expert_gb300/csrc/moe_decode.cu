// The grouped MoE decode layer: grouped gate/up GEMV with SwiGLU + q8_1 of H
// fused into its epilogue, then the grouped down GEMV with the weighted top-k
// combine fused into its epilogue (#242 What it does: native_gu_kernel /
// native_down_kernel over every entry of an expert group; #1525 Change:
// swiglu_quant and the moe_combine sum in slot order).
//
// Two kernels, no host synchronisation:
//  1. gate/up: every CTA rebuilds the expert groups from the routing ids and
//     quantises the layer input (both tiny), then streams work units of one
//     expert x 32 intermediate indices (32 gate rows + the 32 matching up
//     rows), so the SwiGLU and the 32-value q8_1 block of H are finished in
//     the CTA; H itself is never stored, only Hq (workspace).
//  2. down: every CTA owns a contiguous range of output rows across all the
//     routed experts, so it can form out[t] = sum_k w[t,k] * o[(t,k)] for its
//     rows in slot order without any cross-CTA reduction.  Its weight stream
//     depends only on the routing, so it starts before the gate/up kernel has
//     finished (programmatic dependent launch); Hq is read after
//     griddepcontrol.wait.
#include <cuda_fp16.h>

#include "common.cuh"
#include "gemv_core.cuh"
#include "internal.h"

namespace moex {

constexpr int MAX_ENTRIES = 64;   // T * k
constexpr int MAX_GROUP = 8;      // entries per pass of one expert

struct DecodeArgs {
  // gate/up stack [E][2I][H]
  const uint8_t* gu_qs;
  const uint8_t* gu_sc;
  int gu_qrow, gu_scrow;
  // down stack [E][H][I]
  const uint8_t* dn_qs;
  const uint8_t* dn_sc;
  int dn_qrow, dn_scrow;
  int H, I, E, T, k, n;
  const float* x;
  const int32_t* ids;
  const float* w;
  float* out;
  const float* residual;  // nullptr, or added to the combine (may equal out)
  int8_t* hq;      // [n][I]
  float* hds;      // [n][I/32][2]
  float* gu_dbg;
  float* h_dbg;
  int8_t* hq_dbg;
  float* hds_dbg;
  uint32_t* status;
  int nst, stage_bytes;
};

// Expert groups of the routing entries: group g holds entries
// ent[gstart[g] .. gstart[g+1]) (ascending entry index) of expert gexp[g];
// experts ascending; an expert with more than MAX_GROUP entries gets several
// consecutive groups.  Entries with an id outside [0, E) are left out and
// flagged.
struct Groups {
  int ng;
  int gexp[MAX_ENTRIES];
  int gstart[MAX_ENTRIES + 1];
  int ent[MAX_ENTRIES];
};

// Builds the groups from a shared-memory copy of the ids with every thread
// of the block (n <= 64): entry j's position in (expert, entry) order is the
// number of entries before it in that order; a group starts where the expert
// changes or every MAX_GROUP entries of one expert.  The starts are then
// numbered by one warp with ballots over the 64 positions.  Must be called
// by all threads (at least 64); ends with __syncthreads().
__device__ void build_groups(Groups& G, const int32_t* ids, int n, int E, uint32_t* status, int* scratch) {
  // scratch: [MAX_ENTRIES] valid-position map
  const int j = threadIdx.x;
  int e = -1;
  if (j < n) {
    e = ids[j];
    if (e < 0 || e >= E) {
      flag_status(status, DEV_BAD_ROUTE);
      e = -1;
    }
  }
  int pos = -1, run = 0;
  if (e >= 0) {
    pos = 0;
    for (int i = 0; i < n; ++i) {
      const int ei = ids[i];
      if (ei < 0 || ei >= E) continue;
      if (ei < e || (ei == e && i < j)) ++pos;
      if (ei < e) ++run;
    }
    G.ent[pos] = j;
  }
  // by position: the expert of a group starting there, -2 for another
  // valid entry, -1 past the valid entries
  if (j < MAX_ENTRIES) scratch[j] = -1;
  __syncthreads();
  if (e >= 0) scratch[pos] = ((pos - run) % MAX_GROUP == 0) ? e : -2;
  __syncthreads();
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    const int s0 = scratch[lane], s1 = scratch[lane + 32];
    const unsigned st0 = __ballot_sync(0xffffffffu, s0 >= 0), st1 = __ballot_sync(0xffffffffu, s1 >= 0);
    const unsigned v0 = __ballot_sync(0xffffffffu, s0 != -1), v1 = __ballot_sync(0xffffffffu, s1 != -1);
    const unsigned below = (1u << lane) - 1u;
    if (s0 >= 0) {
      const int g = __popc(st0 & below);
      G.gexp[g] = s0;
      G.gstart[g] = lane;
    }
    if (s1 >= 0) {
      const int g = __popc(st0) + __popc(st1 & below);
      G.gexp[g] = s1;
      G.gstart[g] = lane + 32;
    }
    if (lane == 0) {
      const int ng = __popc(st0) + __popc(st1);
      G.gstart[ng] = __popc(v0) + __popc(v1);
      G.ng = ng;
    }
  }
  __syncthreads();
}

// ============================================================== gate / up


constexpr int NUB = 3;    // unit buffers (SwiGLU inputs of one unit)

struct GuSmem {
  int bars, cnt, useq, ucnt, abort_flag, ids, groups, xs, xd, red, ubuf, ring, total;
  __host__ __device__ GuSmem(int T, int H, int NS, int nst, int slot_bytes) {
    const int NB = H / QK;
    int o = 0;
    bars = o; o += 16 * nst;
    cnt = o; o += 4 * nst;
    useq = o; o += 4 * NUB;
    ucnt = o; o += 4 * NUB;
    abort_flag = o; o += 16;
    ids = o; o += 8 * MAX_ENTRIES;
    o = (o + 15) & ~15;
    groups = o; o += static_cast<int>(sizeof(Groups));
    o = (o + 15) & ~15;
    xs = o; o += T * H;
    o = (o + 15) & ~15;
    xd = o; o += 4 * T * NB;
    o = (o + 15) & ~15;
    red = o; o += 4 * NUB * 64 * NS * MAX_GROUP;   // per unit buffer: [64 rows][NS][C]
    ubuf = red;
    o = (o + 127) & ~127;
    ring = o; o += nst * slot_bytes;
    total = o;
  }
};

// SwiGLU + q8_1 of one 32-index block of H for C entries, by one warp:
// lane i takes element i; amax and sum(q) are exact warp reductions, so the
// block is the same as q8_1_block on the same H values.
// g and u are first summed over the K slices, in slice order, from the unit
// buffer ub[row][ks][c] (rows 0..31 gate, 32..63 up).
template <int C>
__device__ __forceinline__ void gu_epilogue(const DecodeArgs& a, const Groups& G, int g, int ib, const float* ub,
                                            int NS, int lane) {
  const int base = G.gstart[g];
#pragma unroll
  for (int c = 0; c < C; ++c) {
    const int j = G.ent[base + c];
    float gv = ub[(lane * NS + 0) * C + c];
    float uv = ub[((32 + lane) * NS + 0) * C + c];
    for (int ks = 1; ks < NS; ++ks) {
      gv = gv + ub[(lane * NS + ks) * C + c];
      uv = uv + ub[((32 + lane) * NS + ks) * C + c];
    }
    const float silu = __fdiv_rn(gv, 1.0f + expf(-gv));
    const float h = __fmul_rn(silu, uv);
    float amax = fabsf(h);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const float d = __fdiv_rn(amax, 127.0f);
    const int q = amax > 0.f ? static_cast<int>(roundf(__fdiv_rn(h, d))) : 0;
    int sum = q;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    const int i = ib * QK + lane;
    a.hq[static_cast<int64_t>(j) * a.I + i] = static_cast<int8_t>(q);
    const float dd = amax > 0.f ? d : 0.f;
    const float ss = amax > 0.f ? __fmul_rn(d, static_cast<float>(sum)) : 0.f;
    if (lane == 0) reinterpret_cast<float2*>(a.hds)[static_cast<int64_t>(j) * (a.I / QK) + ib] = make_float2(dd, ss);
    if (a.gu_dbg) {
      a.gu_dbg[static_cast<int64_t>(j) * 2 * a.I + i] = gv;
      a.gu_dbg[static_cast<int64_t>(j) * 2 * a.I + a.I + i] = uv;
    }
    if (a.h_dbg) a.h_dbg[static_cast<int64_t>(j) * a.I + i] = h;
    if (a.hq_dbg) a.hq_dbg[static_cast<int64_t>(j) * a.I + i] = static_cast<int8_t>(q);
    if (a.hds_dbg && lane == 0)
      reinterpret_cast<float2*>(a.hds_dbg)[static_cast<int64_t>(j) * (a.I / QK) + ib] = make_float2(dd, ss);
  }
}

// Shared state of one decode CTA's consumer loop.
struct StageCtx {
  TmaRing R;
  int nwc, NS, NB;
  int* cnt;
  volatile int* abort_flag;
  float* red;
  uint32_t* status;
};

__device__ __forceinline__ void ctx_abort(const StageCtx& S, int lane, bool& dead) {
  if (lane == 0) {
    *S.abort_flag = 1;
    flag_status(S.status, DEV_TIMEOUT_PIPE);
  }
  dead = true;
}

// One work unit (group g, intermediate block ib): 8 stages of 8 rows, stage
// indices ui*8 .. ui*8+7.  Each warp writes its slice's sums of the unit's
// 64 rows into the unit buffer; the last warp to finish the unit runs the
// SwiGLU + q8_1 epilogue (no hand-off per stage).
template <int C, int WPS>
__device__ __forceinline__ void gu_unit(const DecodeArgs& a, const Groups& G, int g, int ib, int ui,
                                        const StageCtx& S, const ConsumerPos& pos, const int8_t* xs, const float* xd,
                                        int* ucnt, volatile int* useq, float* ubuf, bool& dead) {
  ActRegs<MOEX_Q8_0, C> act;
  {
    const int8_t* xcol[C];
    const float* dcol[C];
#pragma unroll
    for (int c = 0; c < C; ++c) {
      const int t = G.ent[G.gstart[g] + c] / a.k;
      xcol[c] = xs + t * a.H;
      dcol[c] = xd + t * S.NB;
    }
    const int b = pos.ks * SLICE + pos.li;
    load_act<MOEX_Q8_0, C>(act, xcol, dcol, b, b < S.NB, pos.li, 1, smem_half_swap<MOEX_Q8_0>(pos.li));
  }
  constexpr int N = Vals<C, WPS>::N;
  float* ub = ubuf + (ui % NUB) * 64 * S.NS * MAX_GROUP;
  if (!red_slot_wait(&useq[ui % NUB], ui, S.abort_flag)) {
    ctx_abort(S, pos.lane, dead);
    return;
  }
  for (int s = 0; s < 8; ++s) {
    const int it = ui * 8 + s;
    float v[N];
    if (!tma_ring_partials<MOEX_Q8_0, C, WPS, N, true>(S.R, it, pos, SR, S.NB, act, v, S.abort_flag)) {
      ctx_abort(S, pos.lane, dead);
      return;
    }
    reduce_to_red<C, WPS, N>(v, pos, SR, S.NS, ub + s * SR * S.NS * C);
    tma_ring_release(S.R, it, pos.lane);
  }
  int old = 0;
  __syncwarp();
  if (pos.lane == 0) {
    __threadfence_block();
    old = atomicAdd(&ucnt[ui % NUB], 1);
  }
  old = __shfl_sync(0xffffffffu, old, 0);
  if (old == S.nwc - 1) {  // last warp of the unit: SwiGLU + q8_1
    __threadfence_block();
    gu_epilogue<C>(a, G, g, ib, ub, S.NS, pos.lane);
    __syncwarp();
    if (pos.lane == 0) {
      ucnt[ui % NUB] = 0;
      __threadfence_block();
      useq[ui % NUB] = ui + NUB;
    }
  }
}

template <int WPS, int MAXT>
__global__ void __launch_bounds__(MAXT, 1) moe_gu_kernel(DecodeArgs a) {
  extern __shared__ __align__(1024) uint8_t smem[];
  MOEX_TRACE_BEGIN();
  const int NB = a.H / QK;
  const int NS = num_slices(NB);
  const int nwc = NS * WPS;
  const GuSmem L(a.T, a.H, NS, a.nst, a.stage_bytes);
  StageCtx S;
  S.R.full = reinterpret_cast<uint64_t*>(smem + L.bars);
  S.R.empty = S.R.full + a.nst;
  S.R.slots = smem + L.ring;
  S.R.nst = a.nst;
  S.R.slot_bytes = a.stage_bytes;
  S.R.qrow = a.gu_qrow;
  S.R.scrow = a.gu_scrow;
  S.R.slot_rows = SR;
  S.nwc = nwc;
  S.NS = NS;
  S.NB = NB;
  S.cnt = reinterpret_cast<int*>(smem + L.cnt);
  S.abort_flag = reinterpret_cast<volatile int*>(smem + L.abort_flag);
  S.red = reinterpret_cast<float*>(smem + L.red);
  S.status = a.status;
  volatile int* useq = reinterpret_cast<volatile int*>(smem + L.useq);
  int* ucnt = reinterpret_cast<int*>(smem + L.ucnt);
  int32_t* ids_s = reinterpret_cast<int32_t*>(smem + L.ids);
  Groups& G = *reinterpret_cast<Groups*>(smem + L.groups);
  int8_t* xs = reinterpret_cast<int8_t*>(smem + L.xs);
  float* xd = reinterpret_cast<float*>(smem + L.xd);
  float* ubuf = reinterpret_cast<float*>(smem + L.ubuf);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < a.nst; ++i) {
      mbar_init(&S.R.full[i], 1);
      mbar_init(&S.R.empty[i], nwc);
      S.cnt[i] = 0;
    }
    for (int i = 0; i < NUB; ++i) {
      ucnt[i] = 0;
      useq[i] = i;
    }
    *S.abort_flag = 0;
    fence_mbar_init();
  }
  MOEX_TRACE_STAMP(0);
  pdl_wait();  // routing ids and the layer input come from earlier kernels
  MOEX_TRACE_STAMP(1);
  for (int j = threadIdx.x; j < a.n; j += blockDim.x) ids_s[j] = a.ids[j];
  __syncthreads();
  build_groups(G, ids_s, a.n, a.E, a.status, ids_s + MAX_ENTRIES);
  MOEX_TRACE_STAMP(2);
  pdl_launch_dependents();  // after the wait: the routing ids are complete

  const int ib_per = a.I / QK;
  const int units = G.ng * ib_per;
  const int nunit = units > static_cast<int>(blockIdx.x) ? (units - blockIdx.x + gridDim.x - 1) / gridDim.x : 0;

  if (warp == nwc) {
    // the weight stream starts as soon as the groups are known
    if (lane == 0) {
      const uint64_t pol = l2_evict_first_policy();
      int issued = 0;
      for (int ui = 0; ui < nunit && !*S.abort_flag; ++ui) {
        const int u = blockIdx.x + ui * gridDim.x;
        const int g = u / ib_per, ib = u % ib_per;
        const int64_t mat_row0 = static_cast<int64_t>(G.gexp[g]) * 2 * a.I;
        for (int s = 0; s < 8; ++s) {
          const int it = ui * 8 + s;
          const int64_t r0 = mat_row0 + (s < 4 ? ib * QK + s * SR : a.I + ib * QK + (s - 4) * SR);
          if (!tma_ring_fill(S.R, it, a.gu_qs + r0 * a.gu_qrow, a.gu_sc + r0 * a.gu_scrow, SR, pol, S.abort_flag)) {
            *S.abort_flag = 1;
            flag_status(a.status, DEV_TIMEOUT_PIPE);
            break;
          }
          issued = it + 1;
        }
      }
      if (*S.abort_flag)
        for (int it = max(0, issued - a.nst); it < issued; ++it)
          mbar_wait(&S.R.full[it % a.nst], (it / a.nst) & 1, nullptr);
    }
    return;
  }

  // consumers: q8_1 of the layer input (same block arithmetic as quantize_q8_1)
  const int nthr = nwc * 32;
  for (int t = threadIdx.x; t < a.T * NB; t += nthr) {
    const int tok = t / NB, b = t % NB;
    float v[QK];
    const float4* src = reinterpret_cast<const float4*>(a.x + static_cast<int64_t>(tok) * a.H + b * QK);
#pragma unroll
    for (int i = 0; i < QK / 4; ++i) {
      const float4 f = src[i];
      v[4 * i] = f.x; v[4 * i + 1] = f.y; v[4 * i + 2] = f.z; v[4 * i + 3] = f.w;
    }
    uint32_t qw[8];
    float d, s_;
    q8_1_block(v, qw, &d, &s_);
    uint4* dst = reinterpret_cast<uint4*>(xs + tok * a.H + b * QK);
    dst[0] = make_uint4(qw[0], qw[1], qw[2], qw[3]);
    dst[1] = make_uint4(qw[4], qw[5], qw[6], qw[7]);
    xd[tok * NB + b] = d;
  }
  named_bar_sync(1, nthr);

  const ConsumerPos pos = consumer_pos(warp, lane, WPS);
  bool dead = false;
  for (int ui = 0; ui < nunit && !dead; ++ui) {
    const int u = blockIdx.x + ui * gridDim.x;
    const int g = u / ib_per, ib = u % ib_per;
    const int m = G.gstart[g + 1] - G.gstart[g];
#define MOEX_GU(CC) gu_unit<CC, WPS>(a, G, g, ib, ui, S, pos, xs, xd, ucnt, useq, ubuf, dead)
    switch (m) {
      case 1: MOEX_GU(1); break;
      case 2: MOEX_GU(2); break;
      case 3: MOEX_GU(3); break;
      case 4: MOEX_GU(4); break;
      case 5: MOEX_GU(5); break;
      case 6: MOEX_GU(6); break;
      case 7: MOEX_GU(7); break;
      default: MOEX_GU(8); break;
    }
#undef MOEX_GU
    if (ui == 0) MOEX_TRACE_STAMP(3);
  }
  MOEX_TRACE_STAMP(4);
}

// ============================================================== down + combine

struct DnSmem {
  int bars, cnt, abort_flag, ids, groups, red, osum, ring, total;
  __host__ __device__ DnSmem(int n, int I, int NS, int rows_max, int nst, int slot_bytes) {
    (void)I;
    int o = 0;
    bars = o; o += 16 * nst;
    cnt = o; o += 4 * nst;
    abort_flag = o; o += 16;
    ids = o; o += 12 * MAX_ENTRIES;   // ids, build_groups scratch, routing weights
    o = (o + 15) & ~15;
    groups = o; o += static_cast<int>(sizeof(Groups));
    o = (o + 15) & ~15;
    red = o; o += 4 * n * rows_max * NS;   // [entry][row][ks]
    osum = red;
    o = (o + 127) & ~127;
    ring = o; o += nst * slot_bytes;
    total = o;
  }
};

// Stages of one group: the CTA's nrows rows split into ceil(nrows/8) stages
// of balanced size; stage s covers rows [s*nrows/ns, (s+1)*nrows/ns).
__device__ __forceinline__ int dn_nstages(int nrows) { return (nrows + SR - 1) / SR; }

template <int FMT, int C, int WPS>
__device__ __forceinline__ void dn_group(const DecodeArgs& a, const Groups& G, int g, int it0, int nrows,
                                         const StageCtx& S, const ConsumerPos& pos,
                                         float* dred, int rows_max, bool& dead, int c0 = 0, bool release = true) {
  ActRegs<FMT, C> act;
  {
    const int8_t* xcol[C];
    const float* dcol[C];
#pragma unroll
    for (int c = 0; c < C; ++c) {
      const int j = G.ent[G.gstart[g] + c0 + c];
      xcol[c] = a.hq + static_cast<int64_t>(j) * a.I;
      dcol[c] = a.hds + static_cast<int64_t>(j) * S.NB * 2;
    }
    const int b = pos.ks * SLICE + pos.li;
    load_act<FMT, C>(act, xcol, dcol, b, b < S.NB, pos.li, 2, smem_half_swap<FMT>(pos.li));
  }
  constexpr int N = Vals<C, WPS>::N;
  const int gbase = G.gstart[g] + c0;
  // the group's rows arrive as one ring slot; computed 8 rows at a time
  for (int rlo = 0; rlo < nrows; rlo += SR) {
    const int n = nrows - rlo < SR ? nrows - rlo : SR;
    float v[N];
    if (!tma_ring_partials<FMT, C, WPS, N, true>(S.R, it0, pos, n, S.NB, act, v, S.abort_flag, rlo, rlo == 0)) {
      ctx_abort(S, pos.lane, dead);
      return;
    }
    reduce_out<C, WPS, N>(v, pos, n, [&](int row, int c, float val) {
      dred[(G.ent[gbase + c] * rows_max + rlo + row) * S.NS + pos.ks] = val;
    });
  }
  if (release) tma_ring_release(S.R, it0, pos.lane);
}

// TEAMS teams of NS consumer warps (one warp per K slice) take the groups
// round robin, so several groups are in flight at once: a group is little
// work behind a long chain of waits, loads and reductions.
// CMAX == 2: groups are taken two entries at a time, which keeps the kernel
// small enough in registers for ten teams.
template <int FMT, int TEAMS, int MAXT, int CMAX = MAX_GROUP>
__global__ void __launch_bounds__(MAXT, 1) moe_dn_kernel(DecodeArgs a) {
  extern __shared__ __align__(1024) uint8_t smem[];
  MOEX_TRACE_BEGIN();
  const int NB = a.I / QK;
  const int NS = num_slices(NB);
  const int nwc = NS * TEAMS;
  const int G_ = gridDim.x;
  const int rows_max = (a.H + G_ - 1) / G_;
  const DnSmem L(a.n, a.I, NS, rows_max, a.nst, a.stage_bytes);
  StageCtx S;
  S.R.full = reinterpret_cast<uint64_t*>(smem + L.bars);
  S.R.empty = S.R.full + a.nst;
  S.R.slots = smem + L.ring;
  S.R.nst = a.nst;
  S.R.slot_bytes = a.stage_bytes;
  S.R.qrow = a.dn_qrow;
  S.R.scrow = a.dn_scrow;
  S.R.slot_rows = rows_max;
  S.nwc = nwc;
  S.NS = NS;
  S.NB = NB;
  S.cnt = reinterpret_cast<int*>(smem + L.cnt);
  S.abort_flag = reinterpret_cast<volatile int*>(smem + L.abort_flag);
  S.red = reinterpret_cast<float*>(smem + L.red);
  S.status = a.status;
  int32_t* ids_s = reinterpret_cast<int32_t*>(smem + L.ids);
  Groups& G = *reinterpret_cast<Groups*>(smem + L.groups);
  float* osum = reinterpret_cast<float*>(smem + L.osum);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row_begin = static_cast<int>(static_cast<int64_t>(a.H) * blockIdx.x / G_);
  const int row_end = static_cast<int>(static_cast<int64_t>(a.H) * (blockIdx.x + 1) / G_);
  const int nrows = row_end - row_begin;
  const int ns = dn_nstages(nrows);

  if (threadIdx.x == 0) {
    for (int i = 0; i < a.nst; ++i) {
      mbar_init(&S.R.full[i], 1);
      mbar_init(&S.R.empty[i], NS);  // the warps of the team that takes the group
      S.cnt[i] = 0;
    }
    *S.abort_flag = 0;
    fence_mbar_init();
  }
  // The routing ids were complete before the gate/up kernel let this grid
  // launch, so they are read before griddepcontrol.wait.
  float* w_s = reinterpret_cast<float*>(ids_s + 2 * MAX_ENTRIES);  // routing weights, for the combine
  for (int j = threadIdx.x; j < a.n; j += blockDim.x) {
    ids_s[j] = a.ids[j];
    w_s[j] = a.w[j];
  }
  __syncthreads();
  build_groups(G, ids_s, a.n, a.E, nullptr, ids_s + MAX_ENTRIES);
  MOEX_TRACE_STAMP(0);
  pdl_launch_dependents();

  if (warp == nwc) {
    if (lane == 0) {
      const uint64_t pol = l2_evict_first_policy();
      int issued = 0;
      for (int g = 0; g < G.ng; ++g) {
        const int64_t r0 = static_cast<int64_t>(G.gexp[g]) * a.H + row_begin;
        if (!tma_ring_fill(S.R, g, a.dn_qs + r0 * a.dn_qrow, a.dn_sc + r0 * a.dn_scrow, nrows, pol, S.abort_flag)) {
          *S.abort_flag = 1;
          flag_status(a.status, DEV_TIMEOUT_PIPE);
          break;
        }
        issued = g + 1;
      }
      if (*S.abort_flag)
        for (int i = max(0, issued - a.nst); i < issued; ++i) mbar_wait(&S.R.full[i % a.nst], (i / a.nst) & 1, nullptr);
    }
    return;
  }

  // consumers: each team reads its entries' Hq blocks straight from global
  // memory into registers, after the gate/up grid
  pdl_wait();
  MOEX_TRACE_STAMP(1);
  const int nthr = nwc * 32;
  for (int i = threadIdx.x; i < a.n * rows_max * NS; i += nthr) osum[i] = 0.f;
  named_bar_sync(1, nthr);
  const int team = warp / NS;
  const ConsumerPos pos = consumer_pos(warp % NS, lane, 1);
  bool dead = false;
  for (int g = team; g < G.ng && !dead; g += TEAMS) {
    const int m = G.gstart[g + 1] - G.gstart[g];
    if constexpr (CMAX == 2) {
      // entries two at a time (the slot is read again; each entry's dot
      // products are the same bits for any number of columns)
      for (int c0 = 0; c0 < m && !dead; c0 += 2) {
        if (m - c0 >= 2)
          dn_group<FMT, 2, 1>(a, G, g, g, nrows, S, pos, osum, rows_max, dead, c0, c0 + 2 >= m);
        else
          dn_group<FMT, 1, 1>(a, G, g, g, nrows, S, pos, osum, rows_max, dead, c0, true);
      }
    } else {
#define MOEX_DN(CC) dn_group<FMT, CC, 1>(a, G, g, g, nrows, S, pos, osum, rows_max, dead)
      switch (m) {
        case 1: MOEX_DN(1); break;
        case 2: MOEX_DN(2); break;
        case 3: MOEX_DN(3); break;
        case 4: MOEX_DN(4); break;
        case 5: MOEX_DN(5); break;
        case 6: MOEX_DN(6); break;
        case 7: MOEX_DN(7); break;
        default: MOEX_DN(8); break;
      }
#undef MOEX_DN
    }
    if (g == team) MOEX_TRACE_STAMP(2);
  }
  MOEX_TRACE_STAMP(3);
  named_bar_sync(1, nthr);
  // combine: out[t][r] = sum over slots in order of w[t,slot] * o[(t,slot)][r]
  for (int i = threadIdx.x; i < a.T * nrows; i += nthr) {
    const int t = i / nrows, rl = i % nrows;
    float acc = 0.f;
    for (int s = 0; s < a.k; ++s) {
      const int j = t * a.k + s;
      const int e = ids_s[j];
      if (e < 0 || e >= a.E) continue;
      const float* pr = osum + (j * rows_max + rl) * NS;
      float o = pr[0];
      for (int ks = 1; ks < NS; ++ks) o = o + pr[ks];   // slice order, as the dense GEMV
      acc = __fadd_rn(acc, __fmul_rn(w_s[j], o));
    }
    const int64_t o = static_cast<int64_t>(t) * a.H + row_begin + rl;
    a.out[o] = a.residual ? __fadd_rn(a.residual[o], acc) : acc;
  }
  MOEX_TRACE_STAMP(4);
}

// ============================================================== host side

size_t moe_decode_ws_bytes(int T, int k, int64_t hidden, int64_t inter) {
  (void)hidden;
  const size_t n = static_cast<size_t>(T) * k;
  const size_t hq = (n * inter + 255) / 256 * 256;
  return hq + n * (inter / QK) * 8;
}

namespace {

template <int WPS, int MAXT>
moex_status launch_gu(const DecodeArgs& base, int smem_cap, cudaStream_t s) {
  DecodeArgs a = base;
  const int NB = a.H / QK, NS = num_slices(NB);
  const int slot_bytes = ((SR * (a.gu_qrow + a.gu_scrow)) + 127) & ~127;
  a.stage_bytes = slot_bytes;
  int nst = 16;
  for (; nst >= 2; --nst)
    if (GuSmem(a.T, a.H, NS, nst, slot_bytes).total <= smem_cap) break;
  if (nst < 2) return MOEX_EUNSUPPORTED;
  a.nst = nst;
  const GuSmem L(a.T, a.H, NS, nst, slot_bytes);
  auto kern = moe_gu_kernel<WPS, MAXT>;
  if (ensure_smem(reinterpret_cast<const void*>(kern), L.total) != cudaSuccess) return MOEX_ECUDA;
  // grid: enough CTAs for the largest possible unit count is not known on
  // the host (it depends on the routing); use every SM.
  const int grid = sm_count();
  const int threads = (NS * WPS + 1) * 32;
  return cuda_status(launch_pdl(kern, dim3(grid), dim3(threads), L.total, s, a));
}

template <int FMT, int TEAMS, int MAXT, int CMAX = MAX_GROUP>
moex_status launch_dn(const DecodeArgs& base, int smem_cap, cudaStream_t s) {
  DecodeArgs a = base;
  const int NB = a.I / QK, NS = num_slices(NB);
  const int grid = a.H < sm_count() ? a.H : sm_count();
  const int rows_max = (a.H + grid - 1) / grid;
  const int slot_bytes = ((rows_max * (a.dn_qrow + a.dn_scrow)) + 127) & ~127;
  a.stage_bytes = slot_bytes;
  int nst = 16;
  for (; nst >= 2; --nst)
    if (DnSmem(a.n, a.I, NS, rows_max, nst, slot_bytes).total <= smem_cap) break;
  if (nst < 2) return MOEX_EUNSUPPORTED;
  a.nst = nst;
  const DnSmem L(a.n, a.I, NS, rows_max, nst, slot_bytes);
  auto kern = moe_dn_kernel<FMT, TEAMS, MAXT, CMAX>;
  if (ensure_smem(reinterpret_cast<const void*>(kern), L.total) != cudaSuccess) return MOEX_ECUDA;
  const int threads = (NS * TEAMS + 1) * 32;
  return cuda_status(launch_pdl(kern, dim3(grid), dim3(threads), L.total, s, a));
}

// Decode kernels: two warps per K slice up to 8 slices (K <= 4096), else one.
inline int decode_wps(int NS) { return NS <= 3 ? 4 : (NS <= 7 ? 2 : 1); }

template <int FMT>
moex_status launch_dn_fmt(const DecodeArgs& a, int cap, cudaStream_t s) {
  const int NS = num_slices(a.I / QK);
  const int wps = decode_wps(NS);
  if (wps == 4) return launch_dn<FMT, 10, 992, 2>(a, cap, s);  // ten teams of up to three slice warps
  if (wps == 2) return (NS * 2 + 1) * 32 <= 352 ? launch_dn<FMT, 2, 352>(a, cap, s) : launch_dn<FMT, 2, 544>(a, cap, s);
  return (NS + 1) * 32 <= 352 ? launch_dn<FMT, 1, 352>(a, cap, s) : launch_dn<FMT, 1, 544>(a, cap, s);
}

}  // namespace

moex_status launch_moe_decode(const moex_qweight* gu, const moex_qweight* dn, const float* x, int T,
                              const int32_t* ids, const float* w, int k, float* out, void* ws, size_t ws_bytes,
                              float* gu_dbg, float* h_dbg, int8_t* hq_dbg, float* hds_dbg, const float* residual,
                              cudaStream_t s) {
  (void)ws_bytes;
  DecodeArgs a = {};
  a.H = static_cast<int>(gu->K);
  a.I = static_cast<int>(gu->rows / 2);
  a.E = gu->n_mats;
  a.T = T;
  a.k = k;
  a.n = T * k;
  a.gu_qs = static_cast<const uint8_t*>(gu->qs);
  a.gu_sc = static_cast<const uint8_t*>(gu->scales);
  a.gu_qrow = static_cast<int>(qs_row_bytes(gu->fmt, gu->K));
  a.gu_scrow = static_cast<int>(sc_row_bytes(gu->K));
  a.dn_qs = static_cast<const uint8_t*>(dn->qs);
  a.dn_sc = static_cast<const uint8_t*>(dn->scales);
  a.dn_qrow = static_cast<int>(qs_row_bytes(dn->fmt, dn->K));
  a.dn_scrow = static_cast<int>(sc_row_bytes(dn->K));
  a.x = x;
  a.ids = ids;
  a.w = w;
  a.out = out;
  a.residual = residual;
  a.hq = static_cast<int8_t*>(ws);
  a.hds = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + (static_cast<size_t>(a.n) * a.I + 255) / 256 * 256);
  a.gu_dbg = gu_dbg;
  a.h_dbg = h_dbg;
  a.hq_dbg = hq_dbg;
  a.hds_dbg = hds_dbg;
  a.status = device_status_ptr();
  const int cap = max_smem_optin();
  const int NSg = num_slices(a.H / QK), NSd = num_slices(a.I / QK);
  if (NSg > 16 || NSd > 16) return MOEX_EUNSUPPORTED;
  moex_status st;
  if (decode_wps(NSg) == 4)
    st = launch_gu<4, 416>(a, cap, s);
  else if (decode_wps(NSg) == 2)
    st = (NSg * 2 + 1) * 32 <= 352 ? launch_gu<2, 352>(a, cap, s) : launch_gu<2, 544>(a, cap, s);
  else
    st = (NSg + 1) * 32 <= 352 ? launch_gu<1, 352>(a, cap, s) : launch_gu<1, 544>(a, cap, s);
  if (st != MOEX_OK) return st;
  return dn->fmt == MOEX_Q8_0 ? launch_dn_fmt<MOEX_Q8_0>(a, cap, s) : launch_dn_fmt<MOEX_IQ4_NL>(a, cap, s);
}

}  // namespace moex
