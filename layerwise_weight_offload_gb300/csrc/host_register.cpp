// host_register.cpp — all-or-nothing page-locking of host ranges for the
// registered direct H2D transport ([D5] "Registered mmap transport": the
// complete immutable mapped ranges are registered; registration is all or
// nothing, and a rollback that fails leaves mappings that must stay open).
#include <unistd.h>

#include <algorithm>
#include <mutex>
#include <vector>

#include <cuda_runtime.h>

#include "common.h"

namespace dlo {
namespace {

struct Range {
  void* base;
  size_t bytes;
};

// whole pages around [p, p + n)
Range page_range(const void* p, int64_t n) {
  const uintptr_t ps = static_cast<uintptr_t>(sysconf(_SC_PAGESIZE));
  const uintptr_t a = reinterpret_cast<uintptr_t>(p) & ~(ps - 1);
  const uintptr_t b = (reinterpret_cast<uintptr_t>(p) + static_cast<uintptr_t>(n) + ps - 1) &
                      ~(ps - 1);
  return {reinterpret_cast<void*>(a), static_cast<size_t>(b - a)};
}

// fakes for host-side tests of the contract
std::mutex g_fake_mu;
bool g_fake = false;
int32_t g_fail_reg = -1, g_fail_unreg = -1;
int32_t g_reg_calls = 0, g_unreg_calls = 0;
std::vector<int32_t> g_log;

cudaError_t do_register(int32_t i, void* p, size_t n, unsigned flags) {
  {
    std::lock_guard<std::mutex> lock(g_fake_mu);
    if (g_fake) {
      g_log.push_back(i + 1);
      return g_reg_calls++ == g_fail_reg ? cudaErrorInvalidValue : cudaSuccess;
    }
  }
  return cudaHostRegister(p, n, flags);
}

cudaError_t do_unregister(int32_t i, void* p) {
  {
    std::lock_guard<std::mutex> lock(g_fake_mu);
    if (g_fake) {
      g_log.push_back(-(i + 1));
      return g_unreg_calls++ == g_fail_unreg ? cudaErrorInvalidValue : cudaSuccess;
    }
  }
  return cudaHostUnregister(p);
}

// The ranges widened to whole pages, sorted, with the ones that share pages
// merged (CUDA registers a page once).
dlo_status page_ranges(const void* const* ptrs, const int64_t* bytes, int32_t n,
                       std::vector<Range>* out, const char* where) {
  std::vector<Range> rs;
  for (int32_t i = 0; i < n; ++i) {
    if (!ptrs[i] || bytes[i] <= 0)
      DLO_FAIL(DLO_ERR_INVALID, "%s: range %d is empty or null", where, i);
    rs.push_back(page_range(ptrs[i], bytes[i]));
  }
  std::sort(rs.begin(), rs.end(), [](const Range& x, const Range& y) { return x.base < y.base; });
  out->clear();
  for (const Range& r : rs) {
    const uintptr_t b = reinterpret_cast<uintptr_t>(r.base);
    if (!out->empty()) {
      Range& last = out->back();
      const uintptr_t lend = reinterpret_cast<uintptr_t>(last.base) + last.bytes;
      if (b < lend) {
        last.bytes = std::max(lend, b + r.bytes) - reinterpret_cast<uintptr_t>(last.base);
        continue;
      }
    }
    out->push_back(r);
  }
  return DLO_OK;
}

}  // namespace
}  // namespace dlo

extern "C" {

dlo_status dlo_host_register_ranges(const void* const* ptrs, const int64_t* bytes, int32_t n,
                                    int32_t flags, int64_t limit_bytes,
                                    int64_t* registered_bytes) {
  using namespace dlo;
  if (n < 0 || (n > 0 && (!ptrs || !bytes)))
    DLO_FAIL(DLO_ERR_INVALID, "dlo_host_register_ranges: bad arguments");
  std::vector<Range> rs;
  DLO_TRY(page_ranges(ptrs, bytes, n, &rs, "dlo_host_register_ranges"));
  int64_t total = 0;
  for (const Range& r : rs) total += static_cast<int64_t>(r.bytes);
  // preflight: over the ceiling nothing is registered
  if (limit_bytes > 0 && total > limit_bytes)
    DLO_FAIL(DLO_ERR_NOMEM,
             "dlo_host_register_ranges: %lld page-aligned bytes exceed the limit of %lld",
             (long long)total, (long long)limit_bytes);
  unsigned f = cudaHostRegisterPortable | cudaHostRegisterMapped;
  if (flags & 1) f |= cudaHostRegisterReadOnly;
  const int32_t m = static_cast<int32_t>(rs.size());
  for (int32_t i = 0; i < m; ++i) {
    const cudaError_t err = do_register(i, rs[i].base, rs[i].bytes, f);
    if (err == cudaSuccess) continue;
    cudaGetLastError();
    // roll back what this call registered, newest first
    int32_t stuck = 0;
    for (int32_t j = i - 1; j >= 0; --j)
      if (do_unregister(j, rs[j].base) != cudaSuccess) {
        cudaGetLastError();
        ++stuck;
      }
    if (stuck)
      DLO_FAIL(DLO_ERR_PARTIAL,
               "dlo_host_register_ranges: range %d failed (%s) and %d of %d rollbacks failed",
               i, cudaGetErrorString(err), stuck, i);
    DLO_FAIL(DLO_ERR_CUDA, "dlo_host_register_ranges: range %d failed (%s); rolled back", i,
             cudaGetErrorString(err));
  }
  if (registered_bytes) *registered_bytes = total;
  return DLO_OK;
}

dlo_status dlo_host_unregister_ranges(const void* const* ptrs, const int64_t* bytes, int32_t n) {
  using namespace dlo;
  if (n < 0 || (n > 0 && (!ptrs || !bytes)))
    DLO_FAIL(DLO_ERR_INVALID, "dlo_host_unregister_ranges: bad arguments");
  std::vector<Range> rs;
  DLO_TRY(page_ranges(ptrs, bytes, n, &rs, "dlo_host_unregister_ranges"));
  int32_t first_bad = -1;
  cudaError_t bad = cudaSuccess;
  for (int32_t i = 0; i < static_cast<int32_t>(rs.size()); ++i) {
    const cudaError_t err = do_unregister(i, rs[i].base);
    if (err != cudaSuccess && first_bad < 0) {
      first_bad = i;
      bad = err;
    }
    cudaGetLastError();
  }
  if (first_bad >= 0)
    DLO_FAIL(DLO_ERR_CUDA, "dlo_host_unregister_ranges: range %d failed (%s)", first_bad,
             cudaGetErrorString(bad));
  return DLO_OK;
}

dlo_status dlo_debug_fake_host_register(int32_t enable, int32_t fail_register_at,
                                        int32_t fail_unregister_at) {
  using namespace dlo;
  std::lock_guard<std::mutex> lock(g_fake_mu);
  g_fake = enable != 0;
  g_fail_reg = fail_register_at;
  g_fail_unreg = fail_unregister_at;
  g_reg_calls = g_unreg_calls = 0;
  g_log.clear();
  return DLO_OK;
}

dlo_status dlo_debug_fake_host_register_log(int32_t* log, int32_t cap, int32_t* n_calls) {
  using namespace dlo;
  if (!n_calls || (cap > 0 && !log))
    DLO_FAIL(DLO_ERR_INVALID, "dlo_debug_fake_host_register_log: null argument");
  std::lock_guard<std::mutex> lock(g_fake_mu);
  *n_calls = static_cast<int32_t>(g_log.size());
  for (int32_t i = 0; i < cap && i < *n_calls; ++i) log[i] = g_log[i];
  return DLO_OK;
}

}  // extern "C"
