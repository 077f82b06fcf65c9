// attention.cu — non-causal softmax attention of the synthetic DiT block.
//
// o[b, t, head j] = softmax_u( q_t . k_u / sqrt(hd) ) v_u, per batch item and
// head, with q, k, v the three hd-wide column blocks of head j inside the
// bf16 qkv buffer [batch*tokens, 3d] and o written bf16 into [batch*tokens, d].
//
// One CTA = 64 queries of one (batch, head), 4 warps x 16 query rows.  K/V
// tiles of 64 keys are staged in shared memory by cp.async, double
// buffered, with an XOR swizzle on 16-byte chunks so ldmatrix reads are
// conflict-free.  Q K^T and P V run on bf16 mma.sync (m16n8k16, fp32
// accumulate).  Softmax is computed online in the exp2 domain: per row a
// running maximum (reduced across the 4 threads holding the row by warp
// shuffles), a running denominator, and a rescale of the output
// accumulator whenever the maximum grows.  Keys past the end are masked to
// -inf; query rows past the end are computed and not stored.
#include <cuda_bf16.h>

#include <mutex>

#include "common.h"
#include "ptx.cuh"

namespace dlo {
namespace {

constexpr int BQ = 64, BKV = 64, ATT_THREADS = 128;

__device__ __forceinline__ void cp_async16(uint32_t saddr, const void* gptr, bool valid) {
  const int n = valid ? 16 : 0;   // 0 source bytes -> 16 zero bytes written
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(saddr), "l"(gptr), "r"(n)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t saddr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(saddr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t saddr, uint32_t& r0, uint32_t& r1,
                                          uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(saddr));
}

__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                               uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&p);
}

// byte offset of (row, 16-byte chunk) in a swizzled tile with HD columns
template <int HD>
__device__ __forceinline__ uint32_t swz(int row, int chunk) {
  return static_cast<uint32_t>(row * (HD * 2) + ((chunk ^ (row & 7)) << 4));
}

// Copies a [64, HD] tile whose row r starts at src + r*ld (elements) into
// swizzled shared memory; rows with index >= valid_rows become zeros.
template <int HD>
__device__ __forceinline__ void load_tile(uint32_t sbase, const uint16_t* src, int64_t ld,
                                          int valid_rows) {
  constexpr int CHUNKS = HD / 8;
  for (int i = threadIdx.x; i < 64 * CHUNKS; i += ATT_THREADS) {
    const int r = i / CHUNKS, c = i % CHUNKS;
    const bool ok = r < valid_rows;
    const uint16_t* g = src + static_cast<int64_t>(ok ? r : 0) * ld + c * 8;
    cp_async16(sbase + swz<HD>(r, c), g, ok);
  }
}

template <int HD>
__global__ void __launch_bounds__(ATT_THREADS)
attention_kernel(const uint16_t* __restrict__ qkv, int64_t tokens, int64_t d, int heads,
                 uint16_t* __restrict__ o, float scale_log2) {
  constexpr int TILE = 64 * HD * 2;        // bytes of one 64-row tile
  constexpr int KSTEPS = HD / 16;          // k16 steps over the head dim
  constexpr int NB_HD = HD / 8;            // n8 blocks of the output
  extern __shared__ __align__(128) uint8_t smem[];
  const uint32_t sQ = smem_u32(smem);
  const uint32_t sK = sQ + TILE;           // 2 buffers
  const uint32_t sV = sK + 2 * TILE;       // 2 buffers

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int q0 = blockIdx.x * BQ;
  const int head = blockIdx.y, b = blockIdx.z;
  const int64_t ld = 3 * d;
  const uint16_t* base = qkv + static_cast<int64_t>(b) * tokens * ld;
  const uint16_t* gq = base + static_cast<int64_t>(q0) * ld + head * HD;
  const uint16_t* gk = base + d + head * HD;
  const uint16_t* gv = base + 2 * d + head * HD;
  const int n_kv = static_cast<int>((tokens + BKV - 1) / BKV);

  load_tile<HD>(sQ, gq, ld, static_cast<int>(tokens - q0));
  load_tile<HD>(sK, gk, ld, static_cast<int>(tokens));
  load_tile<HD>(sV, gv, ld, static_cast<int>(tokens));
  cp_async_commit();

  uint32_t qf[KSTEPS][4];
  float acc[NB_HD][4];
#pragma unroll
  for (int i = 0; i < NB_HD; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
  float m_run[2] = {-INFINITY, -INFINITY};
  float l_run[2] = {0.f, 0.f};
  const int g = lane >> 2, t4 = lane & 3;

  for (int j = 0; j < n_kv; ++j) {
    if (j + 1 < n_kv) {
      const int nb = (j + 1) & 1;
      const int kv0 = (j + 1) * BKV;
      load_tile<HD>(sK + nb * TILE, gk + static_cast<int64_t>(kv0) * ld, ld,
                    static_cast<int>(tokens - kv0));
      load_tile<HD>(sV + nb * TILE, gv + static_cast<int64_t>(kv0) * ld, ld,
                    static_cast<int>(tokens - kv0));
      cp_async_commit();
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    if (j == 0) {
#pragma unroll
      for (int kk = 0; kk < KSTEPS; ++kk) {
        const int row = warp * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
        const int chunk = 2 * kk + (lane >> 4);
        ldsm_x4(sQ + swz<HD>(row, chunk), qf[kk][0], qf[kk][1], qf[kk][2], qf[kk][3]);
      }
    }
    const uint32_t kb = sK + (j & 1) * TILE;
    const uint32_t vb = sV + (j & 1) * TILE;

    // S = Q K^T for this warp's 16 rows x 64 keys
    float s[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i) s[i][0] = s[i][1] = s[i][2] = s[i][3] = 0.f;
#pragma unroll
    for (int kk = 0; kk < KSTEPS; ++kk) {
#pragma unroll
      for (int nb2 = 0; nb2 < 4; ++nb2) {   // pairs of 8-key blocks
        const int key = nb2 * 16 + ((lane >> 4) << 3) + (lane & 7);
        const int chunk = 2 * kk + ((lane >> 3) & 1);
        uint32_t b0, b1, b2, b3;
        ldsm_x4(kb + swz<HD>(key, chunk), b0, b1, b2, b3);
        mma_bf16_16816(s[2 * nb2], qf[kk], b0, b1);
        mma_bf16_16816(s[2 * nb2 + 1], qf[kk], b2, b3);
      }
    }
    // mask keys past the end, move to the exp2 domain, online softmax
    const int kv0 = j * BKV;
    float mx[2] = {m_run[0], m_run[1]};
#pragma unroll
    for (int nb = 0; nb < 8; ++nb) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int key = kv0 + nb * 8 + 2 * t4 + (e & 1);
        float v = s[nb][e] * scale_log2;
        if (key >= tokens) v = -INFINITY;
        s[nb][e] = v;
        mx[e >> 1] = fmaxf(mx[e >> 1], v);
      }
    }
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 1));
      mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 2));
    }
    float corr[2];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      corr[r] = exp2f(m_run[r] - mx[r]);   // m_run = -inf on the first tile -> 0
      m_run[r] = mx[r];
      l_run[r] *= corr[r];
    }
#pragma unroll
    for (int i = 0; i < NB_HD; ++i) {
      acc[i][0] *= corr[0];
      acc[i][1] *= corr[0];
      acc[i][2] *= corr[1];
      acc[i][3] *= corr[1];
    }
    uint32_t pf[4][4];   // P as four m16k16 A fragments
#pragma unroll
    for (int nb = 0; nb < 8; ++nb) {
      const float p0 = exp2f(s[nb][0] - m_run[0]);
      const float p1 = exp2f(s[nb][1] - m_run[0]);
      const float p2 = exp2f(s[nb][2] - m_run[1]);
      const float p3 = exp2f(s[nb][3] - m_run[1]);
      l_run[0] += p0 + p1;
      l_run[1] += p2 + p3;
      pf[nb >> 1][(nb & 1) * 2 + 0] = pack_bf16(p0, p1);
      pf[nb >> 1][(nb & 1) * 2 + 1] = pack_bf16(p2, p3);
    }
    // O += P V
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
#pragma unroll
      for (int nd2 = 0; nd2 < NB_HD / 2; ++nd2) {
        const int key = kk * 16 + ((lane >> 3) & 1) * 8 + (lane & 7);
        const int chunk = 2 * nd2 + (lane >> 4);
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(vb + swz<HD>(key, chunk), b0, b1, b2, b3);
        mma_bf16_16816(acc[2 * nd2], pf[kk], b0, b1);
        mma_bf16_16816(acc[2 * nd2 + 1], pf[kk], b2, b3);
      }
    }
    __syncthreads();
  }

  // finish the row sums across the quad and store
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    l_run[r] += __shfl_xor_sync(0xffffffffu, l_run[r], 1);
    l_run[r] += __shfl_xor_sync(0xffffffffu, l_run[r], 2);
  }
  const float inv0 = 1.f / l_run[0], inv1 = 1.f / l_run[1];
  const int r0 = q0 + warp * 16 + g, r1 = r0 + 8;
  uint16_t* ob = o + static_cast<int64_t>(b) * tokens * d + head * HD;
#pragma unroll
  for (int i = 0; i < NB_HD; ++i) {
    const int col = i * 8 + 2 * t4;
    if (r0 < tokens)
      *reinterpret_cast<uint32_t*>(ob + static_cast<int64_t>(r0) * d + col) =
          pack_bf16(acc[i][0] * inv0, acc[i][1] * inv0);
    if (r1 < tokens)
      *reinterpret_cast<uint32_t*>(ob + static_cast<int64_t>(r1) * d + col) =
          pack_bf16(acc[i][2] * inv1, acc[i][3] * inv1);
  }
}

template <int HD>
constexpr int att_smem() { return 5 * 64 * HD * 2; }   // Q + 2 K + 2 V tiles

cudaError_t g_att_err = cudaSuccess;
std::once_flag g_att_once;

void set_att_attrs() {
  std::call_once(g_att_once, [] {
    cudaError_t e0 = cudaFuncSetAttribute(attention_kernel<64>,
                                          cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          att_smem<64>());
    cudaError_t e1 = cudaFuncSetAttribute(attention_kernel<128>,
                                          cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          att_smem<128>());
    g_att_err = e0 != cudaSuccess ? e0 : e1;
  });
}

template <int HD>
dlo_status launch_hd(const uint16_t* qkv, int64_t batch, int64_t tokens, int64_t d,
                     int64_t heads, uint16_t* o, cudaStream_t stream) {
  constexpr int SMEM = att_smem<HD>();
  set_att_attrs();
  DLO_CUDA(g_att_err);
  const float scale_log2 = 1.4426950408889634f / sqrtf(static_cast<float>(HD));
  dim3 grid(static_cast<unsigned>((tokens + BQ - 1) / BQ), static_cast<unsigned>(heads),
            static_cast<unsigned>(batch));
  attention_kernel<HD><<<grid, ATT_THREADS, SMEM, stream>>>(qkv, tokens, d,
                                                            static_cast<int>(heads), o,
                                                            scale_log2);
  DLO_CUDA(cudaGetLastError());
  return DLO_OK;
}

}  // namespace

dlo_status attention_preload() {
  set_att_attrs();
  DLO_CUDA(g_att_err);
  return DLO_OK;
}

dlo_status launch_attention(const uint16_t* qkv, int64_t batch, int64_t tokens, int64_t d,
                            int64_t heads, uint16_t* o, cudaStream_t stream) {
  if (batch == 0 || tokens == 0) return DLO_OK;
  if (!qkv || !o || batch < 0 || tokens < 0 || d <= 0 || heads <= 0 || d % heads != 0)
    DLO_FAIL(DLO_ERR_INVALID, "attention: bad arguments (d %lld, heads %lld)", (long long)d,
             (long long)heads);
  if ((reinterpret_cast<uintptr_t>(qkv) | reinterpret_cast<uintptr_t>(o)) & 15u)
    DLO_FAIL(DLO_ERR_INVALID, "attention: qkv and o must be 16-byte aligned");
  if (tokens > (1LL << 31) - BQ || batch > 65535 || heads > 65535)
    DLO_FAIL(DLO_ERR_INVALID, "attention: extent too large");
  const int64_t hd = d / heads;
  if (hd == 64) return launch_hd<64>(qkv, batch, tokens, d, heads, o, stream);
  if (hd == 128) return launch_hd<128>(qkv, batch, tokens, d, heads, o, stream);
  DLO_FAIL(DLO_ERR_INVALID, "attention: head dim %lld not supported (64 or 128)", (long long)hd);
}

}  // namespace dlo
