// status.cu — the device-side error word of the library's kernels.
//
// Every spin-wait inside a kernel is bounded; a wait that runs out writes a
// code (see ptx.cuh, DeviceError) here with atomicCAS so the first failure
// is kept, and the kernel returns early.  The host reads and clears it with
// dlo_kernel_status().
#include <mutex>

#include "common.h"

namespace dlo {

__device__ int g_device_error;

namespace {
std::mutex g_mu;
int* g_addr[64] = {nullptr};
}

int* device_error_word() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) return nullptr;
    g_addr[dev] = static_cast<int*>(p);
  }
  return g_addr[dev];
}

}  // namespace dlo

extern "C" dlo_status dlo_kernel_status(int32_t* code) {
  if (!code) DLO_FAIL(DLO_ERR_INVALID, "dlo_kernel_status: null argument");
  int* w = dlo::device_error_word();
  if (!w) DLO_FAIL(DLO_ERR_CUDA, "dlo_kernel_status: cannot resolve the device error word");
  DLO_CUDA(cudaDeviceSynchronize());
  int v = 0;
  DLO_CUDA(cudaMemcpy(&v, w, sizeof(int), cudaMemcpyDeviceToHost));
  const int zero = 0;
  DLO_CUDA(cudaMemcpy(w, &zero, sizeof(int), cudaMemcpyHostToDevice));
  *code = v;
  return DLO_OK;
}
