// copy_kernel.cu — host->device copy-and-reassemble of one block's shards.
//
// "Distributed Layerwise Offload" (vLLM blog preview, 2026-07-30), "Weight
// Sharding + AllGather", steps 1-2: each rank's shard is copied host->device
// and all_gather_into_tensor places the shards, in rank order, into the
// full-block buffer.  With every shard in this process's pinned host memory,
// both steps become one pass: SMs read each mapped pinned shard over the
// host link with 16-byte loads and write it straight to its final offset
// base_g + r * shard_bytes_g of the slot.
//
// The shard byte length is S_g * esize, which need not be a multiple of 16
// (3 shards of 2731 f32 are 10924 bytes), so a shard's destination may start
// at any byte.  Sources are 16-byte aligned (the ABI requires it) and each
// source buffer holds whole 16-byte words (shard_alloc_bytes).  For a
// destination misaligned by a bytes, the first 16 - a bytes go byte-wise,
// then each aligned 16-byte destination word is assembled from two
// consecutive aligned source words with a funnel shift; lane i takes word
// i+1 from lane i+1 by shuffle, so each source word crosses the link once
// (the last lane of a warp loads its extra word itself).  The last < 16
// bytes go byte-wise.
#include "common.h"

namespace dlo {
namespace {

constexpr int kCopyThreads = 256;

template <int Q>
__device__ __forceinline__ uint4 shift_words(const uint4& w0, const uint4& w1, uint32_t rbits) {
  const uint32_t a[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
  uint4 o;
  o.x = __funnelshift_r(a[Q + 0], a[Q + 1], rbits);
  o.y = __funnelshift_r(a[Q + 1], a[Q + 2], rbits);
  o.z = __funnelshift_r(a[Q + 2], a[Q + 3], rbits);
  o.w = __funnelshift_r(a[Q + 3], a[Q + 4], rbits);
  return o;
}

__device__ __forceinline__ uint4 ld_host16(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// Copies n aligned destination words.  Destination word j receives source
// bytes [h + 16 j, h + 16 j + 16) where h = 4*Q + rbits/8 (0 <= h < 16).
template <int Q>
__device__ __forceinline__ void copy_words(const uint4* __restrict__ src, uint4* __restrict__ dst,
                                           int64_t n, uint32_t rbits, int64_t warp0,
                                           int64_t n_warps, int lane) {
  const bool aligned = (Q == 0 && rbits == 0);
  for (int64_t base = warp0 * 32; base < n; base += n_warps * 32) {
    const int64_t j = base + lane;
    const bool active = j < n;
    uint4 w = make_uint4(0, 0, 0, 0);
    if (active) w = ld_host16(src + j);
    if (aligned) {
      if (active) dst[j] = w;
      continue;
    }
    uint4 nx;
    nx.x = __shfl_down_sync(0xffffffffu, w.x, 1);
    nx.y = __shfl_down_sync(0xffffffffu, w.y, 1);
    nx.z = __shfl_down_sync(0xffffffffu, w.z, 1);
    nx.w = __shfl_down_sync(0xffffffffu, w.w, 1);
    if (active) {
      // lane 31 has no right neighbour; the last word's neighbour is past
      // the body (still inside the 16-byte-rounded source buffer)
      if (lane == 31 || j + 1 >= n) nx = ld_host16(src + j + 1);
      dst[j] = shift_words<Q>(w, nx, rbits);
    }
  }
}

__global__ void __launch_bounds__(kCopyThreads)
copy_reassemble_kernel(const __grid_constant__ SegmentTable t) {
  const int lane = threadIdx.x & 31;
  const int64_t n_warps = static_cast<int64_t>(gridDim.x) * (kCopyThreads / 32);
  const int64_t my_warp = static_cast<int64_t>(blockIdx.x) * (kCopyThreads / 32) + (threadIdx.x >> 5);
  int64_t rot = 0;   // rotates the first warp of each segment to balance work
  for (int s = 0; s < t.n; ++s) {
    const Segment sg = t.seg[s];
    const uint8_t* src = static_cast<const uint8_t*>(sg.src);
    uint8_t* dst = static_cast<uint8_t*>(sg.dst);
    const uint32_t mis = static_cast<uint32_t>(reinterpret_cast<uintptr_t>(dst) & 15u);
    const int64_t head = mis ? (sg.bytes < 16 - mis ? sg.bytes : 16 - mis) : 0;
    const int64_t n_words = (sg.bytes - head) / 16;
    const int64_t tail0 = head + 16 * n_words;
    const int64_t warp0 = (my_warp + rot) % n_warps;
    if (n_words > 0) {
      const uint4* s16 = reinterpret_cast<const uint4*>(src);   // aligned source words
      uint4* d16 = reinterpret_cast<uint4*>(dst + head);        // aligned destination words
      const uint32_t h = static_cast<uint32_t>(head);
      const uint32_t rbits = (h & 3u) * 8u;
      switch (h >> 2) {
        case 0: copy_words<0>(s16, d16, n_words, rbits, warp0, n_warps, lane); break;
        case 1: copy_words<1>(s16, d16, n_words, rbits, warp0, n_warps, lane); break;
        case 2: copy_words<2>(s16, d16, n_words, rbits, warp0, n_warps, lane); break;
        default: copy_words<3>(s16, d16, n_words, rbits, warp0, n_warps, lane); break;
      }
    }
    // byte-wise head and tail, by the warp that would take word 0
    if (warp0 == 0) {
      if (lane < head) dst[lane] = src[lane];
      if (tail0 + lane < sg.bytes) dst[tail0 + lane] = src[tail0 + lane];
    }
    rot = (rot + (n_words + 31) / 32) % n_warps;
  }
}

}  // namespace

dlo_status copy_preload() {
  cudaFuncAttributes attr;
  DLO_CUDA(cudaFuncGetAttributes(&attr, copy_reassemble_kernel));
  return DLO_OK;
}

dlo_status launch_copy_reassemble(const SegmentTable& t, int ctas, cudaStream_t stream) {
  if (t.n <= 0) return DLO_OK;
  if (ctas <= 0) ctas = 152;
  copy_reassemble_kernel<<<ctas, kCopyThreads, 0, stream>>>(t);
  DLO_CUDA(cudaGetLastError());
  return DLO_OK;
}

}  // namespace dlo
