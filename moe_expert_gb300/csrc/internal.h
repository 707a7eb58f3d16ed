// Host-side declarations shared by the moex translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "../../include/moex.h"

namespace moex {

// Device status word of the current device (lazily looked up per device).
uint32_t* device_status_ptr();
int sm_count();
int max_smem_optin();

// Launches a kernel with programmatic stream serialisation allowed, so it
// may start while the previous kernel in the stream drains (kernels call
// griddepcontrol.wait before touching anything the previous kernel writes).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// Raises the dynamic shared-memory limit of a kernel once per device.
cudaError_t ensure_smem(const void* func, size_t bytes);

// The driver's cuTensorMapEncodeTiled (looked up once through the runtime's
// entry-point query, so no link against libcuda), or nullptr.
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn encode_tiled_fn();

inline moex_status cuda_status(cudaError_t e) { return e == cudaSuccess ? MOEX_OK : MOEX_ECUDA; }

// Launchers (argument checks happen in the C entry points).
moex_status launch_quantize_q8_1(const float* x, int64_t K, int ncols, int64_t ldx, int8_t* q, float* ds,
                                 cudaStream_t s);
moex_status launch_weight_pack(const moex_qweight* w, const void* blocks, cudaStream_t s);
moex_status launch_route_topk(const float* logits, int T, int E, int k, int32_t* ids, float* w, cudaStream_t s);
moex_status launch_qgemv(const moex_qweight* W, const int8_t* xq, const float* xds, int ncols, float* y,
                         int64_t ldy, cudaStream_t s);
moex_status launch_qgemv_starved(const moex_qweight* W, const int8_t* xq, const float* xds, int ncols, float* y,
                                 int64_t ldy, uint64_t wait_ns, cudaStream_t s);
moex_status launch_block_dots(const moex_qweight* W, const int8_t* xq, int ncols, int32_t* dots, cudaStream_t s);
size_t moe_decode_ws_bytes(int T, int k, int64_t hidden, int64_t inter);
moex_status launch_moe_decode(const moex_qweight* gu, const moex_qweight* dn, const float* x, int T,
                              const int32_t* ids, const float* w, int k, float* out, void* ws, size_t ws_bytes,
                              float* gu_dbg, float* h_dbg, int8_t* hq_dbg, float* hds_dbg, const float* residual,
                              cudaStream_t s);

// Host checks of the decode layer's arguments (every check of
// moex_moe_decode, in its order, the workspace size last but one).
moex_status check_decode(const moex_qweight* gate_up, const moex_qweight* down, const float* x, int T,
                         const int32_t* ids, const float* w, int k, float* out, void* ws, size_t ws_bytes);

size_t moe_prefill_ws_bytes(int T, int k, int E, int64_t hidden, int64_t inter);
void prefill_ws_layout(int T, int k, int E, int64_t hidden, int64_t inter, size_t* off);
moex_status launch_moe_prefill(const moex_qweight* gu, const moex_qweight* dn, const uint16_t* x, int T,
                               const int32_t* ids, const float* w, int k, const float* residual, float* out, void* ws,
                               cudaStream_t s);

size_t moe_prefill_q8_ws_bytes(int T, int k, int E, int64_t hidden, int64_t inter);
void prefill_q8_ws_layout(int T, int k, int E, int64_t hidden, int64_t inter, size_t* off);
moex_status launch_moe_prefill_q8(const moex_qweight* gu, const moex_qweight* dn, const uint16_t* x, int T,
                                  const int32_t* ids, const float* w, int k, float* out, void* ws, float* h_dbg,
                                  cudaStream_t s);

size_t dense_prefill_ws_bytes(int T, int64_t rows, int64_t K);
moex_status launch_dense_prefill(const moex_qweight* W, const uint16_t* x, int T, float* y, int64_t ldy, void* ws,
                                 cudaStream_t s);

}  // namespace moex
