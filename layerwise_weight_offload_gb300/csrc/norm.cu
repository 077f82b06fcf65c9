// norm.cu — RMSNorm fused with the adaLN modulation of the synthetic DiT
// block: h = bf16( x / sqrt(mean(x^2) + eps) * g * (1 + scale) + shift ).
// One CTA per row; the row is read twice (the second read hits L1/L2), the
// mean square is reduced in a fixed tree order, so results are deterministic.
#include <cuda_bf16.h>

#include "common.h"

namespace dlo {
namespace {

constexpr int kNormThreads = 256;

__global__ void __launch_bounds__(kNormThreads)
rmsnorm_mod_kernel(const float* __restrict__ x, int64_t d, const float* __restrict__ g,
                   const float* __restrict__ shift, const float* __restrict__ scale, float eps,
                   uint16_t* __restrict__ h) {
  const int64_t row = blockIdx.x;
  const float4* xr = reinterpret_cast<const float4*>(x + row * d);
  const int64_t n4 = d / 4;
  float ss = 0.f;
  for (int64_t i = threadIdx.x; i < n4; i += kNormThreads) {
    const float4 v = xr[i];
    ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
  }
  __shared__ float red[kNormThreads / 32];
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
  __syncthreads();
  if (threadIdx.x < 32) {
    float v = threadIdx.x < kNormThreads / 32 ? red[threadIdx.x] : 0.f;
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (threadIdx.x == 0) red[0] = v;
  }
  __syncthreads();
  const float inv = rsqrtf(red[0] / static_cast<float>(d) + eps);
  const float4* g4 = reinterpret_cast<const float4*>(g);
  const float4* s4 = reinterpret_cast<const float4*>(scale);
  const float4* b4 = reinterpret_cast<const float4*>(shift);
  uint2* hr = reinterpret_cast<uint2*>(h + row * d);
  for (int64_t i = threadIdx.x; i < n4; i += kNormThreads) {
    const float4 v = xr[i], gg = g4[i], sc = s4[i], sh = b4[i];
    const float o0 = v.x * inv * gg.x * (1.f + sc.x) + sh.x;
    const float o1 = v.y * inv * gg.y * (1.f + sc.y) + sh.y;
    const float o2 = v.z * inv * gg.z * (1.f + sc.z) + sh.z;
    const float o3 = v.w * inv * gg.w * (1.f + sc.w) + sh.w;
    __nv_bfloat162 p0 = __floats2bfloat162_rn(o0, o1);
    __nv_bfloat162 p1 = __floats2bfloat162_rn(o2, o3);
    uint2 pk;
    pk.x = *reinterpret_cast<uint32_t*>(&p0);
    pk.y = *reinterpret_cast<uint32_t*>(&p1);
    hr[i] = pk;
  }
}

}  // namespace

dlo_status launch_rmsnorm_mod(const float* x, int64_t rows, int64_t d, const float* g,
                              const float* shift, const float* scale, float eps, uint16_t* h,
                              cudaStream_t stream) {
  if (rows == 0) return DLO_OK;
  if (!x || !g || !shift || !scale || !h || rows < 0 || d <= 0 || d % 4 != 0)
    DLO_FAIL(DLO_ERR_INVALID, "rmsnorm_mod: bad arguments (rows %lld, d %lld)",
             (long long)rows, (long long)d);
  if ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(g) |
       reinterpret_cast<uintptr_t>(shift) | reinterpret_cast<uintptr_t>(scale)) & 15u ||
      reinterpret_cast<uintptr_t>(h) & 7u)
    DLO_FAIL(DLO_ERR_INVALID, "rmsnorm_mod: pointers must be 16-byte (h: 8-byte) aligned");
  if (rows > 0x7fffffffLL) DLO_FAIL(DLO_ERR_INVALID, "rmsnorm_mod: too many rows");
  rmsnorm_mod_kernel<<<static_cast<unsigned>(rows), kNormThreads, 0, stream>>>(x, d, g, shift,
                                                                               scale, eps, h);
  DLO_CUDA(cudaGetLastError());
  return DLO_OK;
}

}  // namespace dlo
