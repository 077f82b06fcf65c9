// forward_noalloc.cu — the block forward for callers that cannot allocate
// device memory.
//
// dlo_forward needs a scratch buffer from its caller.  Some callers cannot
// get one: serving loops that must not allocate once they are warm
// (cudaMalloc and cudaFree may synchronise the whole device and stall every
// stream in flight, which a latency budget cannot absorb), and hosts whose
// device memory is owned by another allocator with a fixed budget, so that
// an extra cudaMalloc would fail or overrun it.  dlo_forward_noalloc takes
// its scratch from a fixed array in this library's own device memory
// instead, so it allocates nothing.
//
// The array is a file-scope __device__ array; every GPU on which this
// library's code is loaded holds it until the process exits.  Host code
// never uses the array's name as an address: on first use on a device, with
// that device current, the host asks the runtime for the array's device
// address (cudaGetSymbolAddress) and keeps it per device.
#include <mutex>

#include "common.h"

namespace dlo {
dlo_status forward_impl(const dlo_dit_cfg* cfg, const dlo_plan* plan, const void* block_base,
                        float* x, void* scratch, size_t scratch_bytes, cudaStream_t stream);

namespace {

// 32 MiB: enough for the scratch of, for example, a 1024-token block of
// hidden size 512 with a 2048-wide MLP (dlo_forward_scratch_bytes gives the
// exact need of a shape).
constexpr size_t kNoAllocScratchBytes = static_cast<size_t>(32) << 20;

__device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_noalloc_mu;
void* g_noalloc_addr[64] = {nullptr};

// Device address of g_noalloc_scratch on the current device (set up once
// per device).
dlo_status noalloc_scratch(void** out) {
  int dev = 0;
  DLO_CUDA(cudaGetDevice(&dev));
  if (dev < 0 || dev >= 64) DLO_FAIL(DLO_ERR_INVALID, "dlo_forward_noalloc: device %d", dev);
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (!g_noalloc_addr[dev]) {
    void* p = nullptr;
    const cudaError_t err = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (err != cudaSuccess || !p)
      DLO_FAIL(DLO_ERR_CUDA, "dlo_forward_noalloc: cudaGetSymbolAddress failed: %s",
               cudaGetErrorString(err));
    g_noalloc_addr[dev] = p;
  }
  *out = g_noalloc_addr[dev];
  return DLO_OK;
}

}  // namespace
}  // namespace dlo

extern "C" dlo_status dlo_forward_noalloc(const dlo_dit_cfg* cfg, const dlo_plan* plan,
                                          const void* block_base, float* x, void* stream) {
  using namespace dlo;
  if (!cfg) DLO_FAIL(DLO_ERR_INVALID, "dlo_forward_noalloc: null config");
  const size_t need = dlo_forward_scratch_bytes(cfg);
  if (need > kNoAllocScratchBytes)
    DLO_FAIL(DLO_ERR_NOMEM,
             "dlo_forward_noalloc: this shape needs %zu bytes of scratch; the library's "
             "static scratch holds %zu (use dlo_forward with a caller buffer)",
             need, kNoAllocScratchBytes);
  void* scratch = nullptr;
  DLO_TRY(noalloc_scratch(&scratch));
  // direct launches: instantiating a CUDA graph may allocate
  dlo_dit_cfg c = *cfg;
  c.flags &= ~static_cast<int32_t>(DLO_FWD_GRAPH);
  return forward_impl(&c, plan, block_base, x, scratch, kNoAllocScratchBytes,
                      static_cast<cudaStream_t>(stream));
}
