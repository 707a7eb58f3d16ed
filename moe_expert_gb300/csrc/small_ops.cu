// The activation quantiser, the GGUF -> planes weight repack and the top-k
// router.
#include <cuda_fp16.h>

#include "common.cuh"
#include "gemv_core.cuh"
#include "internal.h"

namespace moex {

// ----------------------------------------------------------------- q8_1

// One thread per 32-value block (#1525 Change: quantize_mmq_q8_1; the block
// arithmetic is q8_1_block, shared with every fused quantiser).
__global__ void __launch_bounds__(128) quantize_q8_1_kernel(const float* __restrict__ x, int K, int NB, int ncols,
                                                            int64_t ldx, int8_t* __restrict__ q,
                                                            float* __restrict__ ds) {
  pdl_wait();
  pdl_launch_dependents();
  const int t = blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= ncols * NB) return;
  const int c = t / NB, b = t % NB;
  const float4* src = reinterpret_cast<const float4*>(x + c * ldx + static_cast<int64_t>(b) * QK);
  float v[QK];
#pragma unroll
  for (int i = 0; i < QK / 4; ++i) {
    const float4 f = src[i];
    v[4 * i] = f.x; v[4 * i + 1] = f.y; v[4 * i + 2] = f.z; v[4 * i + 3] = f.w;
  }
  uint32_t qw[8];
  float d, s;
  q8_1_block(v, qw, &d, &s);
  uint4* dst = reinterpret_cast<uint4*>(q + static_cast<int64_t>(c) * K + static_cast<int64_t>(b) * QK);
  dst[0] = make_uint4(qw[0], qw[1], qw[2], qw[3]);
  dst[1] = make_uint4(qw[4], qw[5], qw[6], qw[7]);
  reinterpret_cast<float2*>(ds)[static_cast<int64_t>(c) * NB + b] = make_float2(d, s);
}

moex_status launch_quantize_q8_1(const float* x, int64_t K, int ncols, int64_t ldx, int8_t* q, float* ds,
                                 cudaStream_t s) {
  const int NB = static_cast<int>(K / QK);
  const int n = ncols * NB;
  return cuda_status(launch_pdl(quantize_q8_1_kernel, dim3((n + 127) / 128), dim3(128), 0, s, x,
                                static_cast<int>(K), NB, ncols, ldx, q, ds));
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
