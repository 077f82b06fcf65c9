// norm.cu — RMSNorm fused with the adaLN modulation of the synthetic DiT
// block: h = bf16( x / sqrt(mean(x^2) + eps) * g * (1 + scale) + shift ).
// One CTA per row (d <= 8192): every thread loads its float4s of the row
// into registers up front, so x is read from HBM once and all loads are in
// flight together; the mean square is reduced per thread, then by a fixed
// shuffle tree per warp, then over the warps in warp order, so results are
// deterministic.  Wider rows: one warp per row, reading the row twice.
#include <cuda_bf16.h>

#include "common.h"
#include "ptx.cuh"

namespace dlo {
namespace {

constexpr int kNormThreads = 256;            // 8 warps, one row per warp
constexpr int kRowsPerCta = kNormThreads / 32;
constexpr int kRowThreads = 256;             // one row per CTA

// One row per CTA of blockDim.x (a multiple of 32, <= kRowThreads) threads;
// thread t holds float4s t, t + blockDim.x, ... (V of them) of the row.
template <int V>
__global__ void __launch_bounds__(kRowThreads)
rmsnorm_mod_row_kernel(const float* __restrict__ x, int64_t d, const float* __restrict__ g,
                       const float* __restrict__ shift, const float* __restrict__ scale,
                       float eps, uint16_t* __restrict__ h) {
  __shared__ float part[kRowThreads / 32];
  grid_dependency_sync();
  const int64_t row = blockIdx.x;
  const int n4 = static_cast<int>(d / 4);
  const int nt = blockDim.x;
  const float4* xr = reinterpret_cast<const float4*>(x + row * d);
  float4 v[V];
#pragma unroll
  for (int k = 0; k < V; ++k) {
    const int i = threadIdx.x + k * nt;
    v[k] = i < n4 ? xr[i] : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  float ss = 0.f;
#pragma unroll
  for (int k = 0; k < V; ++k) ss += v[k].x * v[k].x + v[k].y * v[k].y + v[k].z * v[k].z +
                                    v[k].w * v[k].w;
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = ss;
  __syncthreads();
  float tot = 0.f;
  for (int w = 0; w < nt / 32; ++w) tot += part[w];
  const float inv = rsqrtf(tot / static_cast<float>(d) + eps);
  const float4* g4 = reinterpret_cast<const float4*>(g);
  const float4* s4 = reinterpret_cast<const float4*>(scale);
  const float4* b4 = reinterpret_cast<const float4*>(shift);
  uint2* hr = reinterpret_cast<uint2*>(h + row * d);
#pragma unroll
  for (int k = 0; k < V; ++k) {
    const int i = threadIdx.x + k * nt;
    if (i < n4) {
      const float4 gg = __ldg(g4 + i), sc = __ldg(s4 + i), sh = __ldg(b4 + i);
      const float o0 = v[k].x * inv * gg.x * (1.f + sc.x) + sh.x;
      const float o1 = v[k].y * inv * gg.y * (1.f + sc.y) + sh.y;
      const float o2 = v[k].z * inv * gg.z * (1.f + sc.z) + sh.z;
      const float o3 = v[k].w * inv * gg.w * (1.f + sc.w) + sh.w;
      __nv_bfloat162 p0 = __floats2bfloat162_rn(o0, o1);
      __nv_bfloat162 p1 = __floats2bfloat162_rn(o2, o3);
      uint2 pk;
      pk.x = *reinterpret_cast<uint32_t*>(&p0);
      pk.y = *reinterpret_cast<uint32_t*>(&p1);
      hr[i] = pk;
    }
  }
}

__global__ void __launch_bounds__(kNormThreads)
rmsnorm_mod_kernel(const float* __restrict__ x, int64_t rows, int64_t d,
                   const float* __restrict__ g, const float* __restrict__ shift,
                   const float* __restrict__ scale, float eps, uint16_t* __restrict__ h) {
  grid_dependency_sync();
  const int lane = threadIdx.x & 31;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * kRowsPerCta + (threadIdx.x >> 5);
  if (row >= rows) return;
  const float4* xr = reinterpret_cast<const float4*>(x + row * d);
  const int64_t n4 = d / 4;
  float ss = 0.f;
  for (int64_t i = lane; i < n4; i += 32) {
    const float4 v = xr[i];
    ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
  }
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  const float inv = rsqrtf(ss / static_cast<float>(d) + eps);
  const float4* g4 = reinterpret_cast<const float4*>(g);
  const float4* s4 = reinterpret_cast<const float4*>(scale);
  const float4* b4 = reinterpret_cast<const float4*>(shift);
  uint2* hr = reinterpret_cast<uint2*>(h + row * d);
  for (int64_t i = lane; i < n4; i += 32) {
    const float4 v = xr[i], gg = __ldg(g4 + i), sc = __ldg(s4 + i), sh = __ldg(b4 + i);
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

// Checkpoint-shaped block, after the QKV linear: for each row and head, q
// and k (bf16 in qkv [rows, 3d], columns [0, d) and [d, 2d)) get an RMSNorm
// over the head's HD values with gains gq / gk (when given), then rotary
// embedding (when log2_base > 0): pair (2i, 2i+1) of the token at position
// p (its index within the batch item) is rotated by p * base^(-2i/HD).  One
// warp per (row, head, q or k); lane l holds elements l*E .. l*E+E-1
// (E = HD/32, even), so each pair sits in one lane.  The angle is formed in
// fp32 (absolute error up to about 1e-3 rad at position 16384, below half a
// bf16 unit of the rotated values); cos and sin come from sincosf.
template <int HD>
__global__ void __launch_bounds__(256)
qk_norm_rope_kernel(uint16_t* __restrict__ qkv, int64_t rows, int tokens, int d, int heads,
                    const float* __restrict__ gq, const float* __restrict__ gk, float eps,
                    float log2_base) {
  constexpr int E = HD / 32;
  grid_dependency_sync();
  const int64_t w = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (w >= rows * heads * 2) return;                 // whole warps leave together
  const int part = static_cast<int>(w & 1);
  const int head = static_cast<int>((w >> 1) % heads);
  const int64_t row = (w >> 1) / heads;
  uint16_t* p = qkv + row * 3 * d + part * d + head * HD + lane * E;
  float v[E];
  if (E == 4) {
    const uint2 u = *reinterpret_cast<const uint2*>(p);
    v[0] = __uint_as_float(u.x << 16);
    v[1] = __uint_as_float(u.x & 0xFFFF0000u);
    v[2] = __uint_as_float(u.y << 16);
    v[3] = __uint_as_float(u.y & 0xFFFF0000u);
  } else {
    const uint32_t u = *reinterpret_cast<const uint32_t*>(p);
    v[0] = __uint_as_float(u << 16);
    v[1] = __uint_as_float(u & 0xFFFF0000u);
  }
  const float* g = part == 0 ? gq : gk;
  if (g) {
    float ss = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) ss += v[e] * v[e];
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    const float inv = rsqrtf(ss / static_cast<float>(HD) + eps);
#pragma unroll
    for (int e = 0; e < E; ++e) v[e] = v[e] * inv * __ldg(g + lane * E + e);
  }
  if (log2_base > 0.f) {
    const float pos = static_cast<float>(row % tokens);
#pragma unroll
    for (int k = 0; k < E / 2; ++k) {
      const int i = lane * (E / 2) + k;              // pair index
      const float theta = exp2f(-2.f * static_cast<float>(i) / static_cast<float>(HD) * log2_base);
      float s, c;
      sincosf(pos * theta, &s, &c);
      const float a0 = v[2 * k], b0 = v[2 * k + 1];
      v[2 * k] = a0 * c - b0 * s;
      v[2 * k + 1] = a0 * s + b0 * c;
    }
  }
  uint32_t pk[E / 2];
#pragma unroll
  for (int k = 0; k < E / 2; ++k) {
    __nv_bfloat162 b = __floats2bfloat162_rn(v[2 * k], v[2 * k + 1]);
    pk[k] = *reinterpret_cast<uint32_t*>(&b);
  }
  if (E == 4)
    *reinterpret_cast<uint2*>(p) = make_uint2(pk[0], pk[E / 2 - 1]);
  else
    *reinterpret_cast<uint32_t*>(p) = pk[0];
}

}  // namespace

dlo_status launch_qk_norm_rope(uint16_t* qkv, int64_t batch, int64_t tokens, int64_t d,
                               int64_t heads, const float* gq, const float* gk, float eps,
                               float rope_base, cudaStream_t stream) {
  if (batch == 0 || tokens == 0) return DLO_OK;
  if (!qkv || batch < 0 || tokens < 0 || heads <= 0 || d <= 0 || d % heads != 0 ||
      (!gq) != (!gk) || !(rope_base >= 0.f))
    DLO_FAIL(DLO_ERR_INVALID, "qk_norm_rope: bad arguments");
  const int64_t hd = d / heads;
  if (hd != 64 && hd != 128) DLO_FAIL(DLO_ERR_INVALID, "qk_norm_rope: head dim %lld", (long long)hd);
  if ((reinterpret_cast<uintptr_t>(qkv) & 15u) ||
      (gq && ((reinterpret_cast<uintptr_t>(gq) | reinterpret_cast<uintptr_t>(gk)) & 15u)))
    DLO_FAIL(DLO_ERR_INVALID, "qk_norm_rope: pointers must be 16-byte aligned");
  if (!gq && rope_base == 0.f) return DLO_OK;
  const int64_t rows = batch * tokens;
  const int64_t warps = rows * heads * 2;
  const int64_t blocks = (warps * 32 + 255) / 256;
  if (blocks > 0x7fffffffLL || tokens > 0x7fffffff || d > 0x7fffffff)
    DLO_FAIL(DLO_ERR_INVALID, "qk_norm_rope: too large");
  const float l2b = rope_base > 0.f ? log2f(rope_base) : 0.f;
  if (hd == 64)
    DLO_CUDA(launch_kernel(qk_norm_rope_kernel<64>, dim3(static_cast<unsigned>(blocks)),
                           dim3(256), 0, stream, 1, qkv, rows, static_cast<int>(tokens),
                           static_cast<int>(d), static_cast<int>(heads), gq, gk, eps, l2b));
  else
    DLO_CUDA(launch_kernel(qk_norm_rope_kernel<128>, dim3(static_cast<unsigned>(blocks)),
                           dim3(256), 0, stream, 1, qkv, rows, static_cast<int>(tokens),
                           static_cast<int>(d), static_cast<int>(heads), gq, gk, eps, l2b));
  return DLO_OK;
}

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
  const int64_t n4 = d / 4;
  if (n4 <= 8 * kRowThreads) {
    if (rows > 0x7fffffffLL) DLO_FAIL(DLO_ERR_INVALID, "rmsnorm_mod: too many rows");
    const int nt = n4 >= kRowThreads ? kRowThreads : static_cast<int>((n4 + 31) / 32 * 32);
    const int64_t per = (n4 + nt - 1) / nt;   // float4s per thread, <= 8
    const dim3 grid(static_cast<unsigned>(rows)), block(static_cast<unsigned>(nt));
    auto kern = per <= 1 ? rmsnorm_mod_row_kernel<1>
                : per <= 2 ? rmsnorm_mod_row_kernel<2>
                : per <= 4 ? rmsnorm_mod_row_kernel<4> : rmsnorm_mod_row_kernel<8>;
    DLO_CUDA(launch_kernel(kern, grid, block, 0, stream, 1, x, d, g, shift, scale, eps, h));
    return DLO_OK;
  }
  const int64_t ctas = (rows + kRowsPerCta - 1) / kRowsPerCta;
  if (ctas > 0x7fffffffLL) DLO_FAIL(DLO_ERR_INVALID, "rmsnorm_mod: too many rows");
  DLO_CUDA(launch_kernel(rmsnorm_mod_kernel, dim3(static_cast<unsigned>(ctas)),
                         dim3(kNormThreads), 0, stream, 1, x, rows, d, g, shift, scale, eps, h));
  return DLO_OK;
}

}  // namespace dlo
