// The activation quantiser, the GGUF -> planes weight repack and the top-k
// router.
#include <cuda_fp16.h>

#include "common.cuh"
#include "gemv_core.cuh"
#include "internal.h"

namespace moex {

// ----------------------------------------------------------------- q8_1

// Eight lanes per 32-value block, four values a lane (#1525 Change:
// quantize_mmq_q8_1).  Same arithmetic as q8_1_block: amax over the block
// (shuffles), d = amax / 127 and every q = roundf(x / d) by IEEE division,
// s = d * (sum of q), an all-zero block giving zeros; each lane stores its
// four quants as one word, so a block's 32 bytes go out in one store.
__global__ void __launch_bounds__(128) quantize_q8_1_kernel(const float* __restrict__ x, int K, int NB, int ncols,
                                                            int64_t ldx, int8_t* __restrict__ q,
                                                            float* __restrict__ ds) {
  pdl_wait();
  pdl_launch_dependents();
  const int t = blockIdx.x * blockDim.x + threadIdx.x;
  const int blk = t >> 3, sub = t & 7;   // block index, lane within the block's group of 8
  const bool valid = blk < ncols * NB;
  const int c = valid ? blk / NB : 0, b = valid ? blk % NB : 0;
  float4 f = make_float4(0.f, 0.f, 0.f, 0.f);
  if (valid) f = reinterpret_cast<const float4*>(x + c * ldx + static_cast<int64_t>(b) * QK)[sub];
  float amax = fmaxf(fmaxf(fabsf(f.x), fabsf(f.y)), fmaxf(fabsf(f.z), fabsf(f.w)));
#pragma unroll
  for (int o = 1; o < 8; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  const float d = __fdiv_rn(amax, 127.0f);
  const float v[4] = {f.x, f.y, f.z, f.w};
  int sum = 0;
  uint32_t packed = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    int qi = 0;
    if (amax > 0.f) qi = static_cast<int>(roundf(__fdiv_rn(v[i], d)));
    sum += qi;
    packed |= (static_cast<uint32_t>(qi) & 0xFFu) << (8 * i);
  }
#pragma unroll
  for (int o = 1; o < 8; o <<= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  if (!valid) return;
  reinterpret_cast<uint32_t*>(q + static_cast<int64_t>(c) * K + static_cast<int64_t>(b) * QK)[sub] = packed;
  if (sub == 0)
    reinterpret_cast<float2*>(ds)[static_cast<int64_t>(c) * NB + b] =
        amax > 0.f ? make_float2(d, __fmul_rn(d, static_cast<float>(sum))) : make_float2(0.f, 0.f);
}

moex_status launch_quantize_q8_1(const float* x, int64_t K, int ncols, int64_t ldx, int8_t* q, float* ds,
                                 cudaStream_t s) {
  const int NB = static_cast<int>(K / QK);
  const int64_t threads = static_cast<int64_t>(ncols) * NB * 8;
  return cuda_status(launch_pdl(quantize_q8_1_kernel, dim3(static_cast<unsigned>((threads + 127) / 128)), dim3(128),
                                0, s, x, static_cast<int>(K), NB, ncols, ldx, q, ds));
}

// ----------------------------------------------------------------- weight pack

// One thread per GGUF block: copies the quants of block b of row r into the
// quant plane and its FP16 scale into the scale plane (#1424 What changed:
// device-side GGUF-block -> planes repack).  Padding of a scale row is zeroed
// by the thread of block 0.
__global__ void weight_pack_kernel(const uint8_t* __restrict__ src, int64_t nrows_total, int NB, int fmt,
                                   uint8_t* __restrict__ qs, uint8_t* __restrict__ sc, int64_t qrow, int64_t scrow) {
  const int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (t >= nrows_total * NB) return;
  const int64_t r = t / NB;
  const int b = static_cast<int>(t % NB);
  const int bsz = fmt == MOEX_Q8_0 ? 34 : 18;
  const int qb = fmt == MOEX_Q8_0 ? 32 : 16;
  const uint8_t* blk = src + t * bsz;
  uint8_t* qd = qs + r * qrow + static_cast<int64_t>(b) * qb;
  for (int i = 0; i < qb; ++i) qd[i] = blk[2 + i];
  uint8_t* sd = sc + r * scrow + 2 * b;
  sd[0] = blk[0];
  sd[1] = blk[1];
  if (b == 0)
    for (int64_t i = 2 * NB; i < scrow; ++i) sc[r * scrow + i] = 0;
}

moex_status launch_weight_pack(const moex_qweight* w, const void* blocks, cudaStream_t s) {
  const int NB = static_cast<int>(w->K / QK);
  const int64_t nrows = static_cast<int64_t>(w->n_mats) * w->rows;
  const int64_t n = nrows * NB;
  const int64_t grid = (n + 255) / 256;
  weight_pack_kernel<<<static_cast<unsigned>(grid), 256, 0, s>>>(
      static_cast<const uint8_t*>(blocks), nrows, NB, w->fmt, static_cast<uint8_t*>(w->qs),
      static_cast<uint8_t*>(w->scales), qs_row_bytes(w->fmt, w->K), sc_row_bytes(w->K));
  return cuda_status(cudaGetLastError());
}

// ----------------------------------------------------------------- router

// One warp per token: k rounds of a warp arg-max over the unselected
// logits (larger value first, the lower expert id on ties), then the softmax
// of the k selected logits with the first (largest) subtracted, summed in
// slot order.
// PER = logits a lane holds (E <= 32 * PER); the host picks the smallest.
template <int PER>
__global__ void __launch_bounds__(128) route_topk_kernel(const float* __restrict__ logits, int T, int E, int k,
                                                         int32_t* __restrict__ ids, float* __restrict__ w) {
  pdl_wait();
  pdl_launch_dependents();
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (warp >= T) return;
  const float* row = logits + static_cast<int64_t>(warp) * E;
  float v[PER];
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    const int e = lane + 32 * i;
    v[i] = e < E ? row[e] : -INFINITY;
  }
  uint32_t taken = 0;  // bit i: lane's element i selected
  float my_v = 0.f;    // lane s keeps the logit and id of selection s
  int my_id = 0;
  for (int s = 0; s < k; ++s) {
    float best = -INFINITY;
    int bid = 0x7fffffff;
#pragma unroll
    for (int i = 0; i < PER; ++i) {
      const int e = lane + 32 * i;
      // ascending e within the lane: ties keep the lower id
      if (e < E && !((taken >> i) & 1u) && (bid == 0x7fffffff || v[i] > best)) {
        best = v[i];
        bid = e;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ob = __shfl_xor_sync(0xffffffffu, best, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bid, o);
      if (oi != 0x7fffffff && (bid == 0x7fffffff || ob > best || (ob == best && oi < bid))) {
        best = ob;
        bid = oi;
      }
    }
    if ((bid & 31) == lane) taken |= 1u << (bid >> 5);
    if (lane == s) {
      my_v = best;
      my_id = bid;
    }
  }
  // softmax over the k selected logits, max (selection 0) subtracted, summed in slot order
  const float m = __shfl_sync(0xffffffffu, my_v, 0);
  const float ex = lane < k ? expf(my_v - m) : 0.f;
  float sum = 0.f;
  for (int s = 0; s < k; ++s) sum = sum + __shfl_sync(0xffffffffu, ex, s);
  if (lane < k) {
    ids[static_cast<int64_t>(warp) * k + lane] = my_id;
    w[static_cast<int64_t>(warp) * k + lane] = __fdiv_rn(ex, sum);
  }
}

moex_status launch_route_topk(const float* logits, int T, int E, int k, int32_t* ids, float* w, cudaStream_t s) {
  const int threads = 128;
  const int grid = (T * 32 + threads - 1) / threads;
  if (E <= 128)
    return cuda_status(launch_pdl(route_topk_kernel<4>, dim3(grid), dim3(threads), 0, s, logits, T, E, k, ids, w));
  if (E <= 256)
    return cuda_status(launch_pdl(route_topk_kernel<8>, dim3(grid), dim3(threads), 0, s, logits, T, E, k, ids, w));
  if (E <= 512)
    return cuda_status(launch_pdl(route_topk_kernel<16>, dim3(grid), dim3(threads), 0, s, logits, T, E, k, ids, w));
  return cuda_status(launch_pdl(route_topk_kernel<32>, dim3(grid), dim3(threads), 0, s, logits, T, E, k, ids, w));
}

}  // namespace moex
