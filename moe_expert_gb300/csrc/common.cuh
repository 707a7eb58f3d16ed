// Shared device helpers for the moex kernels (sm_103a only).
//
// PTX wrappers for mbarriers, bulk (TMA) copies, programmatic dependent
// launch and named barriers; the device status word; the q8_1 block
// quantiser used by every kernel that quantises activations.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/moex.h"

#if defined(__CUDA_ARCH__) && (__CUDA_ARCH__ < 1000)
#error "moex kernels target sm_103a (tcgen05, TMA, griddepcontrol)"
#endif

namespace moex {

constexpr int QK = 32;                 // values per quantisation block

// Bits of the device status word (moex_device_status()).
enum : uint32_t {
  DEV_BAD_ROUTE = 1u,                  // a routing id outside [0, n_experts)
  DEV_TIMEOUT_PIPE = 2u,               // an mbarrier wait of a copy pipeline ran out
  DEV_TIMEOUT_MMA = 4u,                // a tensor-core / TMEM wait ran out
  DEV_BAD_SHAPE = 8u,                  // a shape the kernel cannot take reached it
};

// Every bounded wait gives up after this many nanoseconds of %globaltimer.
constexpr uint64_t WAIT_LIMIT_NS = 2000000000ull;

// ----------------------------------------------------------------- basics

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void flag_status(uint32_t* status, uint32_t bits) {
  if (status) atomicOr(status, bits);
}

// ----------------------------------------------------------------- tracing

// Timeline hooks: compiled to nothing unless MOEX_TRACE is defined (a
// profiling build, which defines moex::g_moex_trace and g_moex_trace_ord
// before including the kernels, records %globaltimer at fixed points of
// each CTA).
#ifdef MOEX_TRACE
#define MOEX_TRACE_BEGIN()                                                         \
  __shared__ unsigned int moex_trace_ord;                                          \
  if (threadIdx.x == 0) moex_trace_ord = atomicAdd(&g_moex_trace_ord[blockIdx.x & 4095], 1u)
#define MOEX_TRACE_STAMP(k)                                                        \
  do {                                                                             \
    if (threadIdx.x == 0 && g_moex_trace && moex_trace_ord < 64)                   \
      g_moex_trace[((size_t)moex_trace_ord * 4096 + (blockIdx.x & 4095)) * 8 + (k)] = moex::global_timer_ns(); \
  } while (0)
#else
#define MOEX_TRACE_BEGIN() \
  do {                     \
  } while (0)
#define MOEX_TRACE_STAMP(k) \
  do {                      \
  } while (0)
#endif

// ----------------------------------------------------------------- mbarrier

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Waits for the phase with the given parity to complete.  Returns false if it
// has not completed within limit_ns (WAIT_LIMIT_NS unless a caller passes a
// shorter limit) or if *abort becomes non-zero.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort,
                                          uint64_t limit_ns = WAIT_LIMIT_NS) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 63u) == 0) {
      if (abort && *abort) return false;
      if (global_timer_ns() - t0 > limit_ns) return false;
    }
  }
}

// ----------------------------------------------------------------- bulk copies

// One contiguous global -> shared copy completing on an mbarrier (transaction
// bytes).  dst, src and bytes must be multiples of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Same, with an L2 evict-first policy for data read exactly once.
__device__ __forceinline__ void bulk_g2s_stream(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                                uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], "
      "%4;" ::"r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// ----------------------------------------------------------------- launch control

// Programmatic dependent launch: wait for the preceding grid's memory.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// Allow the next grid in the stream to start launching.
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// ----------------------------------------------------------------- int8 helpers

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

__device__ __forceinline__ int dp4a(uint32_t a, uint32_t b, int c) {
  return __dp4a(static_cast<int>(a), static_cast<int>(b), c);
}

// ----------------------------------------------------------------- q8_1

// q8_1 of one 32-value block: d = amax/127, q = roundf(x/d) (IEEE FP32
// division, half away from zero), s = d * sum(q); an all-zero block gives
// d = q = s = 0.  Writes the 32 quants as 8 packed words in natural order.
__device__ __forceinline__ void q8_1_block(const float* __restrict__ x, uint32_t* __restrict__ qw, float* d_out,
                                           float* s_out) {
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < QK; ++i) amax = fmaxf(amax, fabsf(x[i]));
  const float d = __fdiv_rn(amax, 127.0f);
  int sum = 0;
#pragma unroll
  for (int w = 0; w < 8; ++w) {
    uint32_t packed = 0;
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      int q = 0;
      if (amax > 0.f) q = static_cast<int>(roundf(__fdiv_rn(x[4 * w + b], d)));
      sum += q;
      packed |= (static_cast<uint32_t>(q) & 0xFFu) << (8 * b);
    }
    qw[w] = packed;
  }
  *d_out = amax > 0.f ? d : 0.f;
  *s_out = amax > 0.f ? __fmul_rn(d, static_cast<float>(sum)) : 0.f;
}

// ----------------------------------------------------------------- IQ4_NL

// The IQ4_NL codebook kvalues_iq4nl as int8, low entries (0..7, negative)
// with bit 7 cleared, high entries (8..15, positive) as they are.
constexpr uint32_t IQ4NL_LO7_0 = 0x3F2D1801u;   // -127,-104,-83,-65 & 0x7f
constexpr uint32_t IQ4NL_LO7_1 = 0x766A5D4Fu;   // -49,-35,-22,-10 & 0x7f
constexpr uint32_t IQ4NL_HI_0 = 0x26190D01u;    // 1,13,25,38
constexpr uint32_t IQ4NL_HI_1 = 0x71594535u;    // 53,69,89,113

// The same codebook as two tables for a split dot product: low entries as
// they are (all negative, so prmt's sign-replicate gives -1 where the index
// is >= 8), high entries plus one (all positive, so the flipped selector gives
// 0 where the index is < 8).  The byte-wise sum of the two lookups is the
// codebook value everywhere, so two dp4a's with the same activations give the
// exact integer dot.
constexpr uint32_t IQ4NL_LO_0 = 0xBFAD9881u;    // -127,-104,-83,-65
constexpr uint32_t IQ4NL_LO_1 = 0xF6EADDCFu;    // -49,-35,-22,-10
constexpr uint32_t IQ4NL_HIP1_0 = 0x271A0E02u;  // 2,14,26,39
constexpr uint32_t IQ4NL_HIP1_1 = 0x725A4636u;  // 54,70,90,114

// Decodes the four 4-bit codebook indices held in the low 16 bits of `sel`
// (nibble k -> output byte k) into four int8 codebook values.
//   lo7: entries 0..7 with bit 7 cleared, 0 where the index is >= 8 (prmt's
//        sign-replicate of a byte whose bit 7 is clear);
//   hi : entries 8..15, 0 where the index is < 8 (flag bit flipped);
//   bit 7 is set exactly where lo7 is non-zero (every low entry has a
//   non-zero low part), restoring the negative values.
__device__ __forceinline__ uint32_t iq4nl_lookup4(uint32_t sel, uint32_t sel_flipped) {
  const uint32_t lo7 = prmt(IQ4NL_LO7_0, IQ4NL_LO7_1, sel);
  const uint32_t hi = prmt(IQ4NL_HI_0, IQ4NL_HI_1, sel_flipped);
  const uint32_t sgn = (lo7 + 0x7F7F7F7Fu) & 0x80808080u;
  return lo7 | hi | sgn;
}

}  // namespace moex
