// moex_moe_decode_noalloc: the grouped MoE decode layer for callers that
// cannot allocate device memory.
//
// moex_moe_decode needs a workspace (the q8_1 rows of H that pass from the
// gate/up kernel to the down kernel).  Some callers have no way to get one:
// code that runs inside another framework's memory pool without an allocator
// hook, plug-ins whose host application forbids device allocations after
// start-up, or programs that must not call cudaMalloc at all on the decode
// path (it synchronises the device and can fail under memory pressure).
// This entry point uses a buffer compiled into the library instead: a
// file-scope __device__ array of NOALLOC_SCRATCH_BYTES bytes that every GPU
// loading the library holds until the process exits.  It allocates nothing.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/moex.h"
#include "internal.h"

namespace {

constexpr size_t NOALLOC_SCRATCH_BYTES = 512 * 1024;

// The shared scratch.  Host code must not pass this symbol to a kernel: on
// the host it only names a stand-in; the device address is looked up below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_dev[kMaxDevices];

// Device address of the scratch on the current device, looked up once per
// device with that device current.  Returns nullptr if the lookup fails.
void* scratch_address() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_dev[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) return nullptr;
    g_scratch_dev[dev] = p;
  }
  return g_scratch_dev[dev];
}

}  // namespace

extern "C" {

moex_status moex_moe_decode_noalloc(const moex_qweight* gate_up, const moex_qweight* down, const float* x, int T,
                                    const int32_t* ids, const float* w, int k, float* out, moex_stream stream) {
  void* scratch = scratch_address();
  if (!scratch) return MOEX_ECUDA;
  // The checks of moex_moe_decode, in its order, with the built-in buffer as
  // the workspace: a malformed call gets the same status it would get there,
  // and a well-formed layer that needs more than the buffer gets
  // MOEX_ENOSPACE.
  const moex_status st = moex::check_decode(gate_up, down, x, T, ids, w, k, out, scratch, NOALLOC_SCRATCH_BYTES);
  if (st != MOEX_OK) return st;
  // Nothing in the scratch has to start at zero: the gate/up kernel writes
  // every byte of it that the down kernel reads.
  return moex_moe_decode(gate_up, down, x, T, ids, w, k, out, scratch, NOALLOC_SCRATCH_BYTES, stream);
}

}  // extern "C"
