// The C entry points: argument validation on the host, then launches on the
// caller's stream.  Nothing here allocates device memory.
#include <cuda_runtime.h>

#include <mutex>
#include <unordered_map>

#include "common.cuh"
#include "gemv_core.cuh"
#include "internal.h"

namespace moex {

// The device status word: bit flags set by kernels that see bad input or a
// bounded wait that ran out; read and cleared by moex_device_status().
__device__ uint32_t g_device_status;

namespace {
constexpr int MAX_DEV = 64;
std::mutex g_mu;
uint32_t* g_status_ptr[MAX_DEV];
int g_sms[MAX_DEV];
int g_smem[MAX_DEV];

int current_device() {
  int d = 0;
  if (cudaGetDevice(&d) != cudaSuccess || d < 0 || d >= MAX_DEV) return 0;
  return d;
}
}  // namespace

uint32_t* device_status_ptr() {
  const int d = current_device();
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_status_ptr[d]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_status) == cudaSuccess) g_status_ptr[d] = static_cast<uint32_t*>(p);
  }
  return g_status_ptr[d];
}

int sm_count() {
  const int d = current_device();
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_sms[d]) {
    int v = 0;
    cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, d);
    g_sms[d] = v > 0 ? v : 1;
  }
  return g_sms[d];
}

int max_smem_optin() {
  const int d = current_device();
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_smem[d]) {
    int v = 0;
    cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, d);
    g_smem[d] = v > 0 ? v : 48 * 1024;
  }
  return g_smem[d];
}

EncodeTiledFn encode_tiled_fn() {
  static std::once_flag once;
  static EncodeTiledFn fn = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

cudaError_t ensure_smem(const void* func, size_t bytes) {
  // The attribute is per function and device; it is raised once to the
  // largest size seen, so calls captured into a CUDA graph after a first
  // (warm-up) call make no attribute call at all.
  static std::mutex mu;
  static std::unordered_map<const void*, size_t> seen[MAX_DEV];
  const int d = current_device();
  std::lock_guard<std::mutex> lk(mu);
  auto it = seen[d].find(func);
  if (it != seen[d].end() && it->second >= bytes) return cudaSuccess;
  const cudaError_t e =
      cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
  if (e == cudaSuccess) seen[d][func] = bytes;
  return e;
}

}  // namespace moex

using namespace moex;

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned8(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 7u) == 0; }

moex_status check_weight(const moex_qweight* w) {
  if (!w || !w->qs || !w->scales) return MOEX_EINVAL;
  if (w->fmt != MOEX_Q8_0 && w->fmt != MOEX_IQ4_NL) return MOEX_EUNSUPPORTED;
  if (w->n_mats < 1 || w->rows < 1 || w->K < QK || w->K % QK != 0) return MOEX_EINVAL;
  if (w->rows > (int64_t(1) << 40) || w->K > (int64_t(1) << 20)) return MOEX_EINVAL;
  if (!aligned16(w->qs) || !aligned16(w->scales)) return MOEX_EALIGN;
  return MOEX_OK;
}

moex_status prefill_checked(const moex_qweight* gate_up, const moex_qweight* down, const uint16_t* x_bf16, int T,
                            const int32_t* ids, const float* w, int k, const float* residual, float* out, void* ws,
                            size_t ws_bytes, moex_stream stream) {
  moex_status st = check_weight(gate_up);
  if (st != MOEX_OK) return st;
  st = check_weight(down);
  if (st != MOEX_OK) return st;

  if (!x_bf16 || !ids || !w || !out || !ws) return MOEX_EINVAL;
  if (T < 1 || k < 1 || k > 16 || static_cast<int64_t>(T) * k > (int64_t(1) << 26)) return MOEX_EINVAL;
  if (gate_up->n_mats != down->n_mats || gate_up->n_mats > 4096) return MOEX_EINVAL;
  if (gate_up->rows % 2 != 0 || down->rows != gate_up->K || down->K != gate_up->rows / 2) return MOEX_EINVAL;
  if (gate_up->K % 128 != 0 || down->K % 64 != 0) return MOEX_EUNSUPPORTED;
  // weight rows are 32-bit tensor-map coordinates
  if (static_cast<int64_t>(gate_up->n_mats) * gate_up->rows > INT32_MAX) return MOEX_EUNSUPPORTED;
  if (ws_bytes < moe_prefill_ws_bytes(T, k, gate_up->n_mats, gate_up->K, down->K)) return MOEX_ENOSPACE;
  if (!aligned16(x_bf16) || !aligned16(ws) || !aligned16(out)) return MOEX_EALIGN;
  if (residual && !aligned16(residual)) return MOEX_EALIGN;
  return launch_moe_prefill(gate_up, down, x_bf16, T, ids, w, k, residual, out, ws, stream);
}

}  // namespace

extern "C" {

const char* moex_status_string(int status) {
  switch (status) {
    case MOEX_OK: return "ok";
    case MOEX_EINVAL: return "invalid argument";
    case MOEX_EALIGN: return "pointer or stride not 16-byte aligned";
    case MOEX_EUNSUPPORTED: return "unsupported format or shape";
    case MOEX_ECUDA: return "CUDA error";
    case MOEX_ETIMEOUT: return "device wait timed out";
    case MOEX_EDEVICE: return "bad input detected on the device";
    case MOEX_ENOSPACE: return "workspace too small";
    default: return "unknown status";
  }
}

int moex_version(void) { return 1; }

moex_status moex_weight_plane_bytes(int fmt, int64_t n_mats, int64_t rows, int64_t K, size_t* qs_bytes,
                                    size_t* scale_bytes) {
  if (fmt != MOEX_Q8_0 && fmt != MOEX_IQ4_NL) return MOEX_EUNSUPPORTED;
  if (n_mats < 1 || rows < 1 || K < QK || K % QK != 0 || !qs_bytes || !scale_bytes) return MOEX_EINVAL;
  *qs_bytes = static_cast<size_t>(n_mats * rows * qs_row_bytes(fmt, K));
  *scale_bytes = static_cast<size_t>(n_mats * rows * sc_row_bytes(K));
  return MOEX_OK;
}

moex_status moex_weight_pack(const moex_qweight* w, const void* gguf_blocks, moex_stream stream) {
  const moex_status st = check_weight(w);
  if (st != MOEX_OK) return st;
  if (!gguf_blocks) return MOEX_EINVAL;
  return launch_weight_pack(w, gguf_blocks, stream);
}

moex_status moex_quantize_q8_1(const float* x, int64_t K, int ncols, int64_t ldx, int8_t* q, float* ds,
                               moex_stream stream) {
  if (!x || !q || !ds) return MOEX_EINVAL;
  if (K < QK || K % QK != 0 || K > (1 << 20) || ncols < 1 || ncols > 64 || ldx < K) return MOEX_EINVAL;
  if (!aligned16(x) || !aligned16(q) || !aligned8(ds) || ldx % 4 != 0) return MOEX_EALIGN;
  return launch_quantize_q8_1(x, K, ncols, ldx, q, ds, stream);
}

moex_status moex_qgemv(const moex_qweight* W, const int8_t* xq, const float* xds, int ncols, float* y,
                       int64_t ldy, moex_stream stream) {
  const moex_status st = check_weight(W);
  if (st != MOEX_OK) return st;
  if (W->n_mats != 1) return MOEX_EINVAL;
  if (!xq || !xds || !y || ncols < 1 || ncols > 64 || ldy < W->rows) return MOEX_EINVAL;
  if (W->rows > (int64_t(1) << 31)) return MOEX_EINVAL;
  if (!aligned16(xq) || !aligned8(xds)) return MOEX_EALIGN;
  return launch_qgemv(W, xq, xds, ncols, y, ldy, stream);
}

moex_status moex_qgemv_block_dots(const moex_qweight* W, const int8_t* xq, int ncols, int32_t* dots,
                                  moex_stream stream) {
  const moex_status st = check_weight(W);
  if (st != MOEX_OK) return st;
  if (W->n_mats != 1 || !xq || !dots || ncols < 1 || ncols > 8) return MOEX_EINVAL;
  if (!aligned16(xq)) return MOEX_EALIGN;
  return launch_block_dots(W, xq, ncols, dots, stream);
}

moex_status moex_debug_qgemv_starved(const moex_qweight* W, const int8_t* xq, const float* xds, int ncols, float* y,
                                     int64_t ldy, uint64_t wait_limit_ns, moex_stream stream) {
  const moex_status st = check_weight(W);
  if (st != MOEX_OK) return st;
  if (W->n_mats != 1) return MOEX_EINVAL;
  if (!xq || !xds || !y || ncols != 1 || ldy < W->rows) return MOEX_EINVAL;
  if (W->rows > (int64_t(1) << 31)) return MOEX_EINVAL;
  if (wait_limit_ns < 100000ull || wait_limit_ns > WAIT_LIMIT_NS) return MOEX_EINVAL;
  if (!aligned16(xq) || !aligned8(xds)) return MOEX_EALIGN;
  return launch_qgemv_starved(W, xq, xds, ncols, y, ldy, wait_limit_ns, stream);
}

moex_status moex_route_topk(const float* logits, int T, int E, int k, int32_t* ids, float* w, moex_stream stream) {
  if (!logits || !ids || !w) return MOEX_EINVAL;
  if (T < 1 || k < 1 || k > 16 || E < k || E > 1024) return MOEX_EINVAL;
  return launch_route_topk(logits, T, E, k, ids, w, stream);
}

size_t moex_moe_decode_workspace_bytes(int T, int k, int64_t hidden, int64_t inter) {
  if (T < 1 || k < 1 || inter < QK || hidden < QK) return 0;
  return moe_decode_ws_bytes(T, k, hidden, inter);
}

}  // extern "C"

namespace moex {

moex_status check_decode(const moex_qweight* gate_up, const moex_qweight* down, const float* x, int T,
                                const int32_t* ids, const float* w, int k, float* out, void* ws, size_t ws_bytes) {
  moex_status st = check_weight(gate_up);
  if (st != MOEX_OK) return st;
  st = check_weight(down);
  if (st != MOEX_OK) return st;
  if (gate_up->fmt != MOEX_Q8_0) return MOEX_EUNSUPPORTED;
  if (!x || !ids || !w || !out || !ws) return MOEX_EINVAL;
  if (T < 1 || T > 8 || k < 1 || k > 8) return MOEX_EINVAL;
  if (gate_up->n_mats != down->n_mats) return MOEX_EINVAL;
  if (gate_up->rows % 2 != 0 || down->rows != gate_up->K || down->K != gate_up->rows / 2) return MOEX_EINVAL;
  if (gate_up->K > 8192 || down->K > 8192) return MOEX_EUNSUPPORTED;
  if (ws_bytes < moe_decode_ws_bytes(T, k, gate_up->K, down->K)) return MOEX_ENOSPACE;
  if (!aligned16(x) || !aligned16(ws)) return MOEX_EALIGN;
  return MOEX_OK;
}

}  // namespace moex

extern "C" {

moex_status moex_moe_decode(const moex_qweight* gate_up, const moex_qweight* down, const float* x, int T,
                            const int32_t* ids, const float* w, int k, float* out, void* ws, size_t ws_bytes,
                            moex_stream stream) {
  const moex_status st = check_decode(gate_up, down, x, T, ids, w, k, out, ws, ws_bytes);
  if (st != MOEX_OK) return st;
  return launch_moe_decode(gate_up, down, x, T, ids, w, k, out, ws, ws_bytes, nullptr, nullptr, nullptr, nullptr,
                           nullptr, stream);
}

moex_status moex_moe_decode_residual(const moex_qweight* gate_up, const moex_qweight* down, const float* x, int T,
                                     const int32_t* ids, const float* w, int k, const float* residual, float* out,
                                     void* ws, size_t ws_bytes, moex_stream stream) {
  const moex_status st = check_decode(gate_up, down, x, T, ids, w, k, out, ws, ws_bytes);
  if (st != MOEX_OK) return st;
  if (!residual) return MOEX_EINVAL;
  if (!aligned16(residual)) return MOEX_EALIGN;
  return launch_moe_decode(gate_up, down, x, T, ids, w, k, out, ws, ws_bytes, nullptr, nullptr, nullptr, nullptr,
                           residual, stream);
}

moex_status moex_moe_decode_debug(const moex_qweight* gate_up, const moex_qweight* down, const float* x, int T,
                                  const int32_t* ids, const float* w, int k, float* out, void* ws,
                                  size_t ws_bytes, float* gu_dbg, float* h_dbg, int8_t* hq_dbg, float* hds_dbg,
                                  moex_stream stream) {
  const moex_status st = check_decode(gate_up, down, x, T, ids, w, k, out, ws, ws_bytes);
  if (st != MOEX_OK) return st;
  return launch_moe_decode(gate_up, down, x, T, ids, w, k, out, ws, ws_bytes, gu_dbg, h_dbg, hq_dbg, hds_dbg,
                           nullptr, stream);
}

size_t moex_moe_prefill_workspace_bytes(int T, int k, int E, int64_t hidden, int64_t inter) {
  if (T < 1 || k < 1 || E < 1 || hidden < 128 || inter < 64) return 0;
  return moe_prefill_ws_bytes(T, k, E, hidden, inter);
}

moex_status moex_moe_prefill_workspace_layout(int T, int k, int E, int64_t hidden, int64_t inter,
                                              size_t* offsets) {
  if (!offsets || T < 1 || k < 1 || E < 1 || hidden < 128 || inter < 64) return MOEX_EINVAL;
  prefill_ws_layout(T, k, E, hidden, inter, offsets);
  return MOEX_OK;
}


size_t moex_dense_prefill_workspace_bytes(int T, int64_t rows, int64_t K) {
  if (T < 1 || rows < 128 || K < 64) return 0;
  return dense_prefill_ws_bytes(T, rows, K);
}

moex_status moex_dense_prefill(const moex_qweight* W, const uint16_t* x_bf16, int T, float* y, int64_t ldy, void* ws,
                               size_t ws_bytes, moex_stream stream) {
  const moex_status st = check_weight(W);
  if (st != MOEX_OK) return st;
  if (W->n_mats != 1) return MOEX_EUNSUPPORTED;
  if (!x_bf16 || !y || !ws || T < 1 || T > (1 << 26) || ldy < W->rows || ldy > INT32_MAX) return MOEX_EINVAL;
  if (W->rows % 128 != 0 || W->K % 64 != 0 || W->rows > INT32_MAX) return MOEX_EUNSUPPORTED;
  if (ws_bytes < dense_prefill_ws_bytes(T, W->rows, W->K)) return MOEX_ENOSPACE;
  if (!aligned16(x_bf16) || !aligned16(ws)) return MOEX_EALIGN;
  return launch_dense_prefill(W, x_bf16, T, y, ldy, ws, stream);
}

size_t moex_moe_prefill_q8_workspace_bytes(int T, int k, int E, int64_t hidden, int64_t inter) {
  if (T < 1 || k < 1 || E < 1 || hidden < 128 || inter < 64) return 0;
  return moe_prefill_q8_ws_bytes(T, k, E, hidden, inter);
}

moex_status moex_moe_prefill_q8_workspace_layout(int T, int k, int E, int64_t hidden, int64_t inter,
                                                 size_t* offsets) {
  if (!offsets || T < 1 || k < 1 || E < 1 || hidden < 128 || inter < 64) return MOEX_EINVAL;
  prefill_q8_ws_layout(T, k, E, hidden, inter, offsets);
  return MOEX_OK;
}

static moex_status prefill_q8_checked(const moex_qweight* gate_up, const moex_qweight* down, const uint16_t* x_bf16,
                                      int T, const int32_t* ids, const float* w, int k, float* out, void* ws,
                                      size_t ws_bytes, float* h_dbg, moex_stream stream) {
  moex_status st = check_weight(gate_up);
  if (st != MOEX_OK) return st;
  st = check_weight(down);
  if (st != MOEX_OK) return st;
  if (!x_bf16 || !ids || !w || !out || !ws) return MOEX_EINVAL;
  if (T < 1 || k < 1 || k > 16 || static_cast<int64_t>(T) * k > (int64_t(1) << 26)) return MOEX_EINVAL;
  if (gate_up->n_mats != down->n_mats || gate_up->n_mats > 4096) return MOEX_EINVAL;
  if (gate_up->rows % 2 != 0 || down->rows != gate_up->K || down->K != gate_up->rows / 2) return MOEX_EINVAL;
  if (gate_up->K % 128 != 0 || down->K % 64 != 0) return MOEX_EUNSUPPORTED;
  if (static_cast<int64_t>(gate_up->n_mats) * gate_up->rows > INT32_MAX) return MOEX_EUNSUPPORTED;
  if (ws_bytes < moe_prefill_q8_ws_bytes(T, k, gate_up->n_mats, gate_up->K, down->K)) return MOEX_ENOSPACE;
  if (!aligned16(x_bf16) || !aligned16(ws) || !aligned16(out)) return MOEX_EALIGN;
  if (h_dbg && !aligned16(h_dbg)) return MOEX_EALIGN;
  return launch_moe_prefill_q8(gate_up, down, x_bf16, T, ids, w, k, out, ws, h_dbg, stream);
}

moex_status moex_moe_prefill_q8(const moex_qweight* gate_up, const moex_qweight* down, const uint16_t* x_bf16, int T,
                                const int32_t* ids, const float* w, int k, float* out, void* ws, size_t ws_bytes,
                                moex_stream stream) {
  return prefill_q8_checked(gate_up, down, x_bf16, T, ids, w, k, out, ws, ws_bytes, nullptr, stream);
}

moex_status moex_moe_prefill_q8_debug(const moex_qweight* gate_up, const moex_qweight* down, const uint16_t* x_bf16,
                                      int T, const int32_t* ids, const float* w, int k, float* out, void* ws,
                                      size_t ws_bytes, float* h_dbg, moex_stream stream) {
  return prefill_q8_checked(gate_up, down, x_bf16, T, ids, w, k, out, ws, ws_bytes, h_dbg, stream);
}

moex_status moex_moe_prefill(const moex_qweight* gate_up, const moex_qweight* down, const uint16_t* x_bf16, int T,
                             const int32_t* ids, const float* w, int k, float* out, void* ws, size_t ws_bytes,
                             moex_stream stream) {
  return prefill_checked(gate_up, down, x_bf16, T, ids, w, k, nullptr, out, ws, ws_bytes, stream);
}

moex_status moex_moe_prefill_residual(const moex_qweight* gate_up, const moex_qweight* down, const uint16_t* x_bf16,
                                      int T, const int32_t* ids, const float* w, int k, const float* residual,
                                      float* out, void* ws, size_t ws_bytes, moex_stream stream) {
  if (!residual) return MOEX_EINVAL;
  return prefill_checked(gate_up, down, x_bf16, T, ids, w, k, residual, out, ws, ws_bytes, stream);
}

moex_status moex_device_status(moex_stream stream, uint32_t* flags) {
  if (!flags) return MOEX_EINVAL;
  *flags = 0;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return MOEX_ECUDA;
  uint32_t* p = device_status_ptr();
  if (!p) return MOEX_ECUDA;
  uint32_t v = 0;
  if (cudaMemcpy(&v, p, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return MOEX_ECUDA;
  if (v != 0) {
    const uint32_t zero = 0;
    if (cudaMemcpy(p, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess) return MOEX_ECUDA;
  }
  *flags = v;
  if (v & (DEV_TIMEOUT_PIPE | DEV_TIMEOUT_MMA)) return MOEX_ETIMEOUT;
  if (v != 0) return MOEX_EDEVICE;
  return MOEX_OK;
}

}  // extern "C"
