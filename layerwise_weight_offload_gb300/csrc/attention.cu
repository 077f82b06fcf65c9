// attention.cu — non-causal softmax attention of the synthetic DiT block on
// the 5th-generation tensor cores.
//
// o[b, t, head j] = softmax_u( q_t . k_u / sqrt(hd) ) v_u per batch item and
// head.  Q and K are the first two hd-wide column blocks of head j in the
// bf16 qkv buffer [batch*tokens, 3d]; V is read transposed, vt[b*d + j*hd +
// c, u] (keys contiguous), which the QKV linear's epilogue writes directly,
// so that both products below take K-major operands.
//
// One CTA = 128 queries of one (batch, head), 6 warps:
//   warp 0     TMA: the Q tile once, then K and V^T tiles of 128 keys into a
//              2-stage ring (full/empty mbarriers);
//   warp 1     allocates 512 TMEM columns and issues tcgen05.mma:
//              S_j = Q K_j^T (M=128, N=128) into one of two TMEM S buffers,
//              then O += P_{j-1} V_{j-1} (M=128, N=hd) into the TMEM O
//              accumulator, so the next S overlaps the softmax of the
//              previous tile;
//   warps 2-5  one thread per query row (its TMEM lane): tcgen05.ld of the
//              S row, mask of keys past the end, running maximum and sum in
//              the exp2 domain, P = exp2(s - m) written as bf16 into a
//              128-byte-swizzled shared tile for the next MMA; at the end
//              O / l is stored as bf16.
// The running maximum is allowed to go stale by up to 2^8 (in the exp2
// domain): O in TMEM is rescaled (tcgen05.ld, multiply, tcgen05.st) only
// when a row's maximum grows by more than 8, which keeps every P <= 256.
// Keys past the end are -inf in S and zero in V (TMA zero fill).  All waits
// are bounded; a wait that runs out records a code in the device error
// word and the kernel returns early.
#include <cuda_bf16.h>

#include <mutex>

#include "common.h"
#include "ptx.cuh"

namespace dlo {
namespace {

constexpr int BQ = 128, BKV = 128, ATT_THREADS = 192;
constexpr uint32_t ATT_TMEM_COLS = 512;
constexpr float kRescaleThreshold = 8.f;   // log2 units

template <int HD>
struct AttLayout {
  static constexpr int Q_BYTES = BQ * HD * 2;          // HD/64 chunks of 128 rows x 128 B
  static constexpr int K_BYTES = BKV * HD * 2;
  static constexpr int V_CHUNK = HD * 128;             // HD rows x 64 keys
  static constexpr int V_BYTES = 2 * V_CHUNK;          // 128 keys
  static constexpr int P_CHUNK = BQ * 128;             // 128 rows x 64 keys
  static constexpr int P_BYTES = 2 * P_CHUNK;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + Q_BYTES;
  static constexpr int OFF_V = OFF_K + 2 * K_BYTES;
  static constexpr int OFF_P = OFF_V + 2 * V_BYTES;
  static constexpr int OFF_BAR = OFF_P + 2 * P_BYTES;
  static constexpr int SMEM = OFF_BAR + 256 + 1024;    // barriers + alignment slack
};

__device__ __forceinline__ void att_fail(int* err, volatile int* abort, int code) {
  atomicCAS(err, 0, *abort ? static_cast<int>(DEV_ABORTED) : code);
  *abort = 1;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&p);
}

template <int HD>
__global__ void __launch_bounds__(ATT_THREADS, 1)
attention_tc_kernel(const __grid_constant__ CUtensorMap tm_qk,
                    const __grid_constant__ CUtensorMap tm_vt, int tokens, int d, int heads,
                    uint16_t* __restrict__ o, float scale_log2, int* err) {
  using L = AttLayout<HD>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = smem + L::OFF_Q;
  uint8_t* sK = smem + L::OFF_K;
  uint8_t* sV = smem + L::OFF_V;
  uint8_t* sP = smem + L::OFF_P;
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + L::OFF_BAR);
  uint64_t* q_full = bar + 0;
  uint64_t* k_full = bar + 1;     // [2]
  uint64_t* v_full = bar + 3;     // [2]
  uint64_t* kv_empty = bar + 5;   // [2]
  uint64_t* s_full = bar + 7;     // [2]
  uint64_t* s_empty = bar + 9;    // [2]
  uint64_t* p_full = bar + 11;    // [2]
  uint64_t* pv_done = bar + 13;
  uint64_t* drain = bar + 14;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + 15);
  volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int q0 = blockIdx.x * BQ;
  const int head = blockIdx.y, b = blockIdx.z;
  const int n_kv = (tokens + BKV - 1) / BKV;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&v_full[s], 1);
      mbar_init(&kv_empty[s], 1);
      mbar_init(&s_full[s], 1);
      mbar_init(&s_empty[s], 4);
      mbar_init(&p_full[s], 4);
    }
    mbar_init(pv_done, 1);
    mbar_init(drain, 1);
    *abort = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_qk);
    tma_prefetch_desc(&tm_vt);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, ATT_TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tS = tmem;             // two buffers of 128 columns
  const uint32_t tO = tmem + 256;       // HD columns

  if (warp == 0) {
    if (lane == 0) {
      const int row_q = b * tokens + q0;
      mbar_arrive_expect_tx(q_full, L::Q_BYTES);
      for (int c = 0; c < HD / 64; ++c)
        tma_load_2d(sQ + c * (BQ * 128), &tm_qk, q_full, head * HD + 64 * c, row_q);
      int issued = 0;
      bool ok = true;
      for (int j = 0; j < n_kv; ++j) {
        const int s = j & 1;
        const uint32_t n = static_cast<uint32_t>(j >> 1);
        if (!mbar_wait_bounded(&kv_empty[s], (n & 1u) ^ 1u, abort)) {
          att_fail(err, abort, DEV_TIMEOUT_PRODUCER);
          ok = false;
          break;
        }
        const int kv0 = j * BKV;
        mbar_arrive_expect_tx(&k_full[s], L::K_BYTES);
        for (int c = 0; c < HD / 64; ++c)
          tma_load_2d(sK + s * L::K_BYTES + c * (BKV * 128), &tm_qk, &k_full[s],
                      d + head * HD + 64 * c, b * tokens + kv0);
        mbar_arrive_expect_tx(&v_full[s], L::V_BYTES);
        for (int c = 0; c < 2; ++c)
          tma_load_2d(sV + s * L::V_BYTES + c * L::V_CHUNK, &tm_vt, &v_full[s], kv0 + 64 * c,
                      (b * heads + head) * HD);
        ++issued;
      }
      if (!ok) {
        // let the copies already issued land before the CTA can exit
        volatile int never = 0;
        mbar_wait_bounded(q_full, 0, &never);
        for (int j = issued - 2 < 0 ? 0 : issued - 2; j < issued; ++j) {
          mbar_wait_bounded(&k_full[j & 1], static_cast<uint32_t>((j >> 1) & 1), &never);
          mbar_wait_bounded(&v_full[j & 1], static_cast<uint32_t>((j >> 1) & 1), &never);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16_f32(BQ, BKV);
      constexpr uint32_t idesc_o = idesc_bf16_f32(BQ, HD);
      bool ok = mbar_wait_bounded(q_full, 0, abort);
      if (!ok) att_fail(err, abort, DEV_TIMEOUT_MMA_FULL);
      const uint32_t q_addr = smem_u32(sQ);
      for (int j = 0; ok && j <= n_kv; ++j) {
        if (j < n_kv) {
          const int s = j & 1;
          const uint32_t n = static_cast<uint32_t>(j >> 1);
          if (!mbar_wait_bounded(&k_full[s], n & 1u, abort) ||
              !mbar_wait_bounded(&s_empty[s], (n & 1u) ^ 1u, abort)) {
            att_fail(err, abort, DEV_TIMEOUT_MMA_FULL);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t k_addr = smem_u32(sK + s * L::K_BYTES);
#pragma unroll
          for (int kk = 0; kk < HD / 16; ++kk) {
            const uint32_t off = (kk >> 2) * (BQ * 128) + (kk & 3) * 32;
            umma_bf16(tS + s * BKV, sdesc_k_sw128(q_addr + off), sdesc_k_sw128(k_addr + off),
                      idesc_s, kk > 0 ? 1u : 0u);
          }
          umma_commit(&s_full[s]);
        }
        if (j >= 1) {
          const int jj = j - 1;
          const int s = jj & 1;
          const uint32_t n = static_cast<uint32_t>(jj >> 1);
          if (!mbar_wait_bounded(&p_full[s], n & 1u, abort) ||
              !mbar_wait_bounded(&v_full[s], n & 1u, abort)) {
            att_fail(err, abort, DEV_TIMEOUT_MMA_FULL);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t p_addr = smem_u32(sP + s * L::P_BYTES);
          const uint32_t v_addr = smem_u32(sV + s * L::V_BYTES);
#pragma unroll
          for (int kk = 0; kk < BKV / 16; ++kk) {
            umma_bf16(tO, sdesc_k_sw128(p_addr + (kk >> 2) * L::P_CHUNK + (kk & 3) * 32),
                      sdesc_k_sw128(v_addr + (kk >> 2) * L::V_CHUNK + (kk & 3) * 32), idesc_o,
                      (jj > 0 || kk > 0) ? 1u : 0u);
          }
          umma_commit(&kv_empty[s]);
          umma_commit(pv_done);
        }
      }
      if (!ok) {
        volatile int never = 0;
        umma_commit(drain);
        mbar_wait_bounded(drain, 0, &never);
      }
    }
  } else {
    const int quad = warp & 3;
    const int row = quad * 32 + lane;          // query row in the tile == TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < n_kv; ++j) {
      const int s = j & 1;
      const uint32_t n = static_cast<uint32_t>(j >> 1);
      if (!__all_sync(0xffffffffu, mbar_wait_bounded(&s_full[s], n & 1u, abort))) {
        if (lane == 0) att_fail(err, abort, DEV_TIMEOUT_EPILOGUE);
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t sr[4][32];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld_32x32b_x32(tS + s * BKV + c * 32 + lane_off, sr[c]);
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&s_empty[s]);
      const int kv0 = j * BKV;
      const int valid = tokens - kv0;          // keys of this tile that exist
      float mt = -INFINITY;
#pragma unroll
      for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          float x = __uint_as_float(sr[c][i]) * scale_log2;
          if (c * 32 + i >= valid) x = -INFINITY;
          sr[c][i] = __float_as_uint(x);
          mt = fmaxf(mt, x);
        }
      if (j == 0) {
        m = mt;
      } else {
        const bool need = mt > m + kRescaleThreshold;
        if (__any_sync(0xffffffffu, need)) {
          // O must hold every product up to tile j-1 before it is scaled
          if (!__all_sync(0xffffffffu,
                          mbar_wait_bounded(pv_done, static_cast<uint32_t>((j - 1) & 1), abort))) {
            if (lane == 0) att_fail(err, abort, DEV_TIMEOUT_EPILOGUE);
            ok = false;
            break;
          }
          tc_fence_after();
          float corr = 1.f;
          if (need) {
            corr = exp2f(m - mt);
            m = mt;
            l *= corr;
          }
#pragma unroll 1
          for (int c = 0; c < HD / 32; ++c) {
            uint32_t orr[32];
            tmem_ld_32x32b_x32(tO + c * 32 + lane_off, orr);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i)
              orr[i] = __float_as_uint(__uint_as_float(orr[i]) * corr);
            tmem_st_32x32b_x32(tO + c * 32 + lane_off, orr);
          }
          tmem_st_wait();
        }
      }
      // P = exp2(s - m) as bf16 into the swizzled P tile of this stage
      uint8_t* prow = sP + s * L::P_BYTES + row * 128;
#pragma unroll
      for (int c = 0; c < 16; ++c) {
        float p[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          p[e] = exp2f(__uint_as_float(sr[c >> 2][(c & 3) * 8 + e]) - m);
          l += p[e];
        }
        const uint4 v = make_uint4(pack_bf16(p[0], p[1]), pack_bf16(p[2], p[3]),
                                   pack_bf16(p[4], p[5]), pack_bf16(p[6], p[7]));
        const int cc = c & 7;
        *reinterpret_cast<uint4*>(prow + (c >> 3) * L::P_CHUNK + ((cc ^ (row & 7)) << 4)) = v;
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[s]);
    }
    if (ok) {
      if (!__all_sync(0xffffffffu,
                      mbar_wait_bounded(pv_done, static_cast<uint32_t>((n_kv - 1) & 1), abort))) {
        if (lane == 0) att_fail(err, abort, DEV_TIMEOUT_EPILOGUE);
      } else {
        tc_fence_after();
        const float inv = 1.f / l;
        const int t = q0 + row;
        uint16_t* orow = o + (static_cast<int64_t>(b) * tokens + t) * d + head * HD;
#pragma unroll 1
        for (int c = 0; c < HD / 32; ++c) {
          uint32_t orr[32];
          tmem_ld_32x32b_x32(tO + c * 32 + lane_off, orr);
          tmem_ld_wait();
          if (t < tokens) {
#pragma unroll
            for (int g = 0; g < 4; ++g) {
              const uint4 v = make_uint4(
                  pack_bf16(__uint_as_float(orr[8 * g + 0]) * inv,
                            __uint_as_float(orr[8 * g + 1]) * inv),
                  pack_bf16(__uint_as_float(orr[8 * g + 2]) * inv,
                            __uint_as_float(orr[8 * g + 3]) * inv),
                  pack_bf16(__uint_as_float(orr[8 * g + 4]) * inv,
                            __uint_as_float(orr[8 * g + 5]) * inv),
                  pack_bf16(__uint_as_float(orr[8 * g + 6]) * inv,
                            __uint_as_float(orr[8 * g + 7]) * inv));
              *reinterpret_cast<uint4*>(orow + c * 32 + 8 * g) = v;
            }
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, ATT_TMEM_COLS);
  }
}

// V block of qkv ([rows, 3d], columns [2d, 3d)) -> vt [b*d + c, t] with row
// stride vt_ld; 64 x 64 tiles through shared memory so that both the reads
// and the writes are coalesced.
__global__ void __launch_bounds__(256)
transpose_v_kernel(const uint16_t* __restrict__ qkv, int tokens, int d, uint16_t* __restrict__ vt,
                   int64_t vt_ld) {
  __shared__ uint16_t tile[64][66];
  const int t0 = blockIdx.x * 64, c0 = blockIdx.y * 64, b = blockIdx.z;
  const uint16_t* src = qkv + static_cast<int64_t>(b) * tokens * 3 * d + 2 * d;
  for (int i = threadIdx.x; i < 64 * 64; i += 256) {
    const int r = i / 64, c = i % 64;           // r: token, c: feature
    const int t = t0 + r;
    tile[r][c] = t < tokens ? src[static_cast<int64_t>(t) * 3 * d + c0 + c] : uint16_t(0);
  }
  __syncthreads();
  for (int i = threadIdx.x; i < 64 * 64; i += 256) {
    const int c = i / 64, r = i % 64;           // c: feature (row of vt), r: token
    const int t = t0 + r;
    if (t < tokens) vt[(static_cast<int64_t>(b) * d + c0 + c) * vt_ld + t] = tile[r][c];
  }
}

cudaError_t g_att_err = cudaSuccess;
std::once_flag g_att_once;

void set_att_attrs() {
  std::call_once(g_att_once, [] {
    cudaError_t e0 = cudaFuncSetAttribute(attention_tc_kernel<64>,
                                          cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          AttLayout<64>::SMEM);
    cudaError_t e1 = cudaFuncSetAttribute(attention_tc_kernel<128>,
                                          cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          AttLayout<128>::SMEM);
    g_att_err = e0 != cudaSuccess ? e0 : e1;
  });
}

template <int HD>
dlo_status launch_hd(const CUtensorMap& tm_qk, const CUtensorMap& tm_vt, int64_t batch,
                     int64_t tokens, int64_t d, int64_t heads, uint16_t* o, int* err,
                     cudaStream_t stream) {
  set_att_attrs();
  DLO_CUDA(g_att_err);
  const float scale_log2 = 1.4426950408889634f / sqrtf(static_cast<float>(HD));
  dim3 grid(static_cast<unsigned>((tokens + BQ - 1) / BQ), static_cast<unsigned>(heads),
            static_cast<unsigned>(batch));
  attention_tc_kernel<HD><<<grid, ATT_THREADS, AttLayout<HD>::SMEM, stream>>>(
      tm_qk, tm_vt, static_cast<int>(tokens), static_cast<int>(d), static_cast<int>(heads), o,
      scale_log2, err);
  DLO_CUDA(cudaGetLastError());
  return DLO_OK;
}

}  // namespace

int64_t vt_ld_for(int64_t tokens) { return (tokens + 7) / 8 * 8; }

dlo_status attention_preload() {
  set_att_attrs();
  DLO_CUDA(g_att_err);
  return DLO_OK;
}

dlo_status launch_attention_vt(const uint16_t* qkv, const uint16_t* vt, int64_t vt_ld,
                               int64_t batch, int64_t tokens, int64_t d, int64_t heads,
                               uint16_t* o, cudaStream_t stream) {
  if (batch == 0 || tokens == 0) return DLO_OK;
  if (!qkv || !vt || !o || batch < 0 || tokens < 0 || d <= 0 || heads <= 0 || d % heads != 0)
    DLO_FAIL(DLO_ERR_INVALID, "attention: bad arguments (d %lld, heads %lld)", (long long)d,
             (long long)heads);
  if ((reinterpret_cast<uintptr_t>(qkv) | reinterpret_cast<uintptr_t>(vt) |
       reinterpret_cast<uintptr_t>(o)) & 15u)
    DLO_FAIL(DLO_ERR_INVALID, "attention: qkv, vt and o must be 16-byte aligned");
  if (batch * tokens > (1LL << 31) - 1 || batch > 65535 || heads > 65535 ||
      vt_ld < tokens || vt_ld % 8 != 0 || batch * d > (1LL << 31) - 1)
    DLO_FAIL(DLO_ERR_INVALID, "attention: extent too large or bad vt row stride");
  const int64_t hd = d / heads;
  if (hd != 64 && hd != 128)
    DLO_FAIL(DLO_ERR_INVALID, "attention: head dim %lld not supported (64 or 128)",
             (long long)hd);
  int* err = device_error_word();
  if (!err) DLO_FAIL(DLO_ERR_CUDA, "attention: cannot resolve the device error word");
  CUtensorMap tm_qk, tm_vt;
  DLO_TRY(make_tmap_2d(&tm_qk, qkv, batch * tokens, 3 * d, 3 * d, BQ, 64));
  DLO_TRY(make_tmap_2d(&tm_vt, vt, batch * d, tokens, vt_ld, static_cast<uint32_t>(hd), 64));
  if (hd == 64) return launch_hd<64>(tm_qk, tm_vt, batch, tokens, d, heads, o, err, stream);
  return launch_hd<128>(tm_qk, tm_vt, batch, tokens, d, heads, o, err, stream);
}

dlo_status launch_transpose_v(const uint16_t* qkv, int64_t batch, int64_t tokens, int64_t d,
                              uint16_t* vt, int64_t vt_ld, cudaStream_t stream) {
  if (batch == 0 || tokens == 0) return DLO_OK;
  if (!qkv || !vt || d % 64 != 0 || vt_ld < tokens)
    DLO_FAIL(DLO_ERR_INVALID, "transpose_v: bad arguments");
  dim3 grid(static_cast<unsigned>((tokens + 63) / 64), static_cast<unsigned>(d / 64),
            static_cast<unsigned>(batch));
  transpose_v_kernel<<<grid, 256, 0, stream>>>(qkv, static_cast<int>(tokens),
                                               static_cast<int>(d), vt, vt_ld);
  DLO_CUDA(cudaGetLastError());
  return DLO_OK;
}

}  // namespace dlo
