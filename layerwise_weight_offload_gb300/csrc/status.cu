// status.cu — the device-side error word of the library's kernels.
//
// Every spin-wait inside a kernel is bounded; a wait that runs out writes a
// code (see ptx.cuh, DeviceError) here with atomicCAS so the first failure
// is kept, and the kernel returns early.  The host reads and clears it with
// dlo_kernel_status().
#include <mutex>

#include "common.h"
#include "ptx.cuh"

namespace dlo {

__device__ int g_device_error;
__device__ unsigned long long g_probe_elapsed_ns;

namespace {

// One CTA of 64 threads.  Thread 0 waits, with the same bounded wait the
// kernels use (suspending or spinning) but limit_ns instead of their
// limit, on phase 0 of an mbarrier on which no thread arrives until the
// wait has returned; thread 32 sets the CTA's abort flag after abort_ns if
// abort_ns > 0 (the path by which one role of a kernel stops the others).
// A wait that gives up records DEV_TIMEOUT_PROBE in the error word; the
// barrier is then completed so that nothing is left pending.
__global__ void wait_probe_kernel(int spin, uint64_t limit_ns, uint64_t abort_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  volatile int* abort = &abort_flag;
  if (threadIdx.x == 0) {
    const uint64_t t0 = globaltimer_ns();
    const bool ok = spin ? mbar_wait_spin(&bar, 0, abort, limit_ns)
                         : mbar_wait_bounded(&bar, 0, abort, limit_ns);
    g_probe_elapsed_ns = globaltimer_ns() - t0;
    if (!ok)
      atomicCAS(&g_device_error, 0, static_cast<int>(*abort ? DEV_ABORTED : DEV_TIMEOUT_PROBE));
    mbar_arrive(&bar);
  } else if (threadIdx.x == 32 && abort_ns > 0) {
    const uint64_t t0 = globaltimer_ns();
    // bounded: abort_ns is at most 2 s (checked on the host)
    while (globaltimer_ns() - t0 < abort_ns) {
    }
    *abort = 1;
  }
  __syncthreads();
}

}  // namespace

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

namespace {
thread_local bool t_pdl_scope = false;
int g_launch_overlap = -1;
}  // namespace

bool pdl_active() { return t_pdl_scope; }
PdlScope::PdlScope(bool on) : prev(t_pdl_scope) { t_pdl_scope = on; }
PdlScope::~PdlScope() { t_pdl_scope = prev; }
int launch_overlap_mode() { return g_launch_overlap; }

}  // namespace dlo

extern "C" dlo_status dlo_set_launch_overlap(int32_t on) {
  if (on < -1 || on > 1) DLO_FAIL(DLO_ERR_INVALID, "dlo_set_launch_overlap: -1, 0 or 1");
  dlo::g_launch_overlap = on;
  return DLO_OK;
}

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

extern "C" dlo_status dlo_debug_wait_probe(int32_t spin, int64_t limit_ns, int64_t abort_ns,
                                           int64_t* elapsed_ns, int32_t* code) {
  using namespace dlo;
  if (!elapsed_ns || !code) DLO_FAIL(DLO_ERR_INVALID, "dlo_debug_wait_probe: null argument");
  if (limit_ns < 0 || limit_ns > 2000000000LL || abort_ns < 0 || abort_ns > 2000000000LL)
    DLO_FAIL(DLO_ERR_INVALID, "dlo_debug_wait_probe: limits must be 0..2 s");
  int32_t before = 0;
  DLO_TRY(dlo_kernel_status(&before));   // start from a clear word
  wait_probe_kernel<<<1, 64>>>(spin ? 1 : 0, static_cast<uint64_t>(limit_ns),
                               static_cast<uint64_t>(abort_ns));
  DLO_CUDA(cudaGetLastError());
  unsigned long long el = 0;
  DLO_CUDA(cudaMemcpyFromSymbol(&el, g_probe_elapsed_ns, sizeof(el)));
  int32_t c = 0;
  DLO_TRY(dlo_kernel_status(&c));
  *elapsed_ns = static_cast<int64_t>(el);
  *code = c;
  if (c != 0) DLO_FAIL(DLO_ERR_TIMEOUT, "dlo_debug_wait_probe: the wait gave up (code %d)", c);
  return DLO_OK;
}
