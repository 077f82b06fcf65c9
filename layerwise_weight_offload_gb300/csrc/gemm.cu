// gemm.cu — the block's linears on the 5th-generation tensor cores.
//
// out = epilogue(A W^T): A bf16 [M, K] (activations, K contiguous), W bf16
// [N, K] (a weight view inside a slot, nn.Linear layout, K contiguous), fp32
// accumulation in tensor memory.  Epilogues: store bf16; GELU-tanh then
// store bf16; gated residual x[M, N] += gate[N] * acc in fp32.
//
// Structure (one CTA per SM, persistent over 128 x 256 output tiles):
//   warp 0     TMA producer: 128x64 A box and 256x64 W box per stage,
//              128-byte swizzled, 4-stage ring guarded by full/empty
//              mbarriers;
//   warp 1     allocates 512 TMEM columns (two 256-column fp32
//              accumulators) and one thread issues tcgen05.mma
//              (M=128, N=256, K=16, kind::f16) and tcgen05.commit;
//   warps 2-5  epilogue: tcgen05.ld of their 32-lane quarter, the fused
//              epilogue, stores to global; they release the accumulator so
//              the next tile's MMAs overlap this tile's epilogue.
// Ragged M, N and K are covered by TMA zero fill and epilogue masks.
// Work units: output tiles, or (tile, K slice) when K is split — for every
// tile when there are too few tiles for the SMs, or only for the tiles of a
// short last wave (the tail), which then spread over the idle SMs.  Split
// units write fp32 partials to a workspace that a second kernel sums in slice
// order before the epilogue.  No atomics: every output element is produced
// by one thread in a fixed order, so results do not depend on addresses or
// scheduling.
// Large linears run instead on pairs of CTAs (gemm_pair_kernel below): one
// tcgen05.mma.cta_group::2 over two SMs per 256 x 256 tile, each CTA loading
// half of both operand tiles; pair_auto chooses between the two kernels.
#include <cuda.h>
#include <cuda_bf16.h>

#include <mutex>

#include "common.h"
#include "ptx.cuh"

namespace dlo {
namespace {

constexpr int BM = 128, BN = 256, BK = 64, STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;          // 16 KB
constexpr int B_BYTES = BN * BK * 2;          // 32 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int NUM_THREADS = 192;
constexpr uint32_t TMEM_COLS = 512;
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 /*align*/ + 256 /*barriers*/;

// Output tile t -> (row block, column block) in groups of group_m row
// blocks, row blocks fastest within a group: the tiles of one wave
// (consecutive t) then cover group_m row blocks by about 152/group_m column
// blocks.  With A larger than L2 this keeps the operands a wave streams
// small (Super's fc2: 16 x 9.5 blocks instead of all 64 row blocks of a
// 403 MB A by 2.4 column blocks, which read A from DRAM ten times); with A
// small enough to stay in L2 one group spans all rows (column-major), so
// that each weight column block is read once.
constexpr int kGroupM = 16;
constexpr int64_t kAResidentBytes = 64ll << 20;
__host__ __device__ __forceinline__ void tile_coords(int t, int num_m, int num_n, int group_m,
                                                     int& m_idx, int& n_idx) {
  const int per_group = group_m * num_n;
  const int first_m = (t / per_group) * group_m;
  const int rows = num_m - first_m < group_m ? num_m - first_m : group_m;
  const int r = t - (t / per_group) * per_group;
  m_idx = first_m + r % rows;
  n_idx = r / rows;
}

__device__ __forceinline__ void record_failure(int* err, volatile int* abort, int code) {
  atomicCAS(err, 0, code);
  *abort = 1;
}

// GELU in its tanh form, 0.5 z (1 + tanh(u)) with u = sqrt(2/pi) (z + 0.044715
// z^3), computed through the identity 0.5 (1 + tanh(u)) = 1 / (1 + e^(-2u)):
// z / (1 + 2^(-2u log2 e)) with the hardware exp2 and reciprocal
// approximations (a few ulp relative, on both tails: the result goes to 0
// for large negative z and to z for large positive z).  The full-precision
// tanhf costs dozens of instructions per element, and four epilogue warps
// doing that saturate the SM sub-partitions that the loader and the MMA
// issuer share with them.
__device__ __forceinline__ float gelu_tanh(float z) {
  const float k0 = 0.7978845608028654f;   // sqrt(2/pi)
  const float k1 = 0.044715f;
  const float m2log2e = -2.8853900817779268f;   // -2 log2(e)
  const float u = k0 * fmaf(k1 * z * z, z, z);
  float e, r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e) : "f"(u * m2log2e));
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(1.f + e));
  return z * r;
}

// r[i] (fp32 bits) += bias[n0 + i] for the columns below N (N a multiple of 8).
__device__ __forceinline__ void add_bias32(uint32_t (&r)[32], const uint16_t* bias, int64_t n0,
                                           int64_t N) {
#pragma unroll
  for (int g = 0; g < 4; ++g) {
    if (n0 + 8 * g + 8 > N) break;
    const uint4 b = __ldg(reinterpret_cast<const uint4*>(bias + n0 + 8 * g));
    const uint32_t w[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      r[8 * g + 2 * e] = __float_as_uint(__uint_as_float(r[8 * g + 2 * e]) +
                                         __uint_as_float(w[e] << 16));
      r[8 * g + 2 * e + 1] = __float_as_uint(__uint_as_float(r[8 * g + 2 * e + 1]) +
                                             __uint_as_float(w[e] & 0xFFFF0000u));
    }
  }
}

template <int EPI>
__device__ __forceinline__ void epilogue_store(const uint32_t (&r)[32], int64_t row, int64_t n0,
                                               int64_t N, int ks, const EpiArgs& ea) {
  void* out = ea.out;
  const float* gate = ea.gate;
  if (EPI == EPI_PARTIAL) {
    // fp32 partial sum of one K slice: ws[ks][row][n0..n0+31]
    float* pr = ea.ws + (static_cast<int64_t>(ks) * ea.ws_rows + row) * N + n0;
#pragma unroll
    for (int g = 0; g < 8; ++g)
      if (n0 + 4 * g + 4 <= N)
        *reinterpret_cast<float4*>(pr + 4 * g) =
            make_float4(__uint_as_float(r[4 * g]), __uint_as_float(r[4 * g + 1]),
                        __uint_as_float(r[4 * g + 2]), __uint_as_float(r[4 * g + 3]));
    return;
  }
  if (EPI == EPI_QKV && n0 >= ea.v_col0) {
    // V columns: transposed store, vt[b*d + c, t]; the 32 lanes of a warp
    // hold 32 consecutive rows, so each store instruction writes 64
    // contiguous bytes of one vt row
    const int64_t b = row / ea.tokens, t = row - b * ea.tokens;
    const int64_t d = ea.v_col0 / 2;
    uint16_t* dst = ea.vt + (b * d + (n0 - ea.v_col0)) * ea.vt_ld + t;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      __nv_bfloat16 v = __float2bfloat16_rn(__uint_as_float(r[i]));
      dst[static_cast<int64_t>(i) * ea.vt_ld] = *reinterpret_cast<uint16_t*>(&v);
    }
    return;
  }
  if (EPI == EPI_RESID_F32) {
    // all eight loads of x (and of the gate) are issued before the first
    // store, so the read-modify-write waits for one memory latency per
    // 32 columns, not eight: with a short K the epilogue is otherwise
    // slower than the next tile's mainloop it should hide behind
    float* xr = static_cast<float*>(out) + row * N + n0;
    float4 xv[8], gv[8];
#pragma unroll
    for (int g = 0; g < 8; ++g)
      if (n0 + 4 * g + 4 <= N) {
        xv[g] = *reinterpret_cast<const float4*>(xr + 4 * g);
        gv[g] = __ldg(reinterpret_cast<const float4*>(gate + n0 + 4 * g));
      }
#pragma unroll
    for (int g = 0; g < 8; ++g) {
      if (n0 + 4 * g + 4 <= N) {
        xv[g].x += gv[g].x * __uint_as_float(r[4 * g + 0]);
        xv[g].y += gv[g].y * __uint_as_float(r[4 * g + 1]);
        xv[g].z += gv[g].z * __uint_as_float(r[4 * g + 2]);
        xv[g].w += gv[g].w * __uint_as_float(r[4 * g + 3]);
        *reinterpret_cast<float4*>(xr + 4 * g) = xv[g];
      }
    }
  } else {
    uint32_t pk[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      float a = __uint_as_float(r[2 * j]), b = __uint_as_float(r[2 * j + 1]);
      if (EPI == EPI_GELU_BF16) {
        a = gelu_tanh(a);
        b = gelu_tanh(b);
      }
      __nv_bfloat162 p = __floats2bfloat162_rn(a, b);
      pk[j] = *reinterpret_cast<uint32_t*>(&p);
    }
    uint16_t* orow = static_cast<uint16_t*>(out) + row * N + n0;
#pragma unroll
    for (int g = 0; g < 4; ++g)
      if (n0 + 8 * g + 8 <= N)
        *reinterpret_cast<uint4*>(orow + 8 * g) =
            make_uint4(pk[4 * g], pk[4 * g + 1], pk[4 * g + 2], pk[4 * g + 3]);
  }
}

template <int EPI>
__global__ void __launch_bounds__(NUM_THREADS, 1)
gemm_tcgen05_kernel(const __grid_constant__ CUtensorMap tma_a,
                    const __grid_constant__ CUtensorMap tma_b, int M, int N, int K,
                    int splits, int tail, int tail_splits, int group_m, const EpiArgs ea,
                    int* err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + STAGES * A_BYTES;
  uint64_t* full = reinterpret_cast<uint64_t*>(sB + STAGES * B_BYTES);
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 4);
    }
    mbar_init(drain, 1);
    *abort = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tma_a);
    tma_prefetch_desc(&tma_b);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  grid_dependency_wait();

  const int num_m = (M + BM - 1) / BM;
  const int num_n = (N + BN - 1) / BN;
  const int num_tiles = num_m * num_n;
  const int num_k = (K + BK - 1) / BK;
  // work units: (tile, K slice of `splits`) for the first num_tiles - tail
  // tiles, then (tail tile, K slice of `tail_splits`); slice ks of nks covers
  // k-blocks [ks num_k / nks, (ks + 1) num_k / nks)
  const int n_main = (num_tiles - tail) * splits;
  const int num_units = n_main + tail * tail_splits;
  auto unit_of = [&](int u, int& tile, int& ks, int& nks, int& tt) {
    if (u < n_main) {
      tile = u / splits;
      ks = u - tile * splits;
      nks = splits;
      tt = -1;
    } else {
      tt = (u - n_main) / tail_splits;
      ks = (u - n_main) - tt * tail_splits;
      nks = tail_splits;
      tile = num_tiles - tail + tt;
    }
  };

  if (warp == 0) {
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int issued = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < num_units && ok; u += gridDim.x) {
        int tile, ks, nks, tt;
        unit_of(u, tile, ks, nks, tt);
        const int kb0 = static_cast<int>(static_cast<int64_t>(ks) * num_k / nks);
        const int kb1 = static_cast<int>(static_cast<int64_t>(ks + 1) * num_k / nks);
        int m_idx, n_idx;
        tile_coords(tile, num_m, num_n, group_m, m_idx, n_idx);
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait_spin(&empty[stage], phase ^ 1u, abort)) {
            record_failure(err, abort, *abort ? DEV_ABORTED : DEV_TIMEOUT_PRODUCER);
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&full[stage], STAGE_BYTES);
          tma_load_2d(sA + stage * A_BYTES, &tma_a, &full[stage], kb * BK, m_idx * BM);
          tma_load_2d(sB + stage * B_BYTES, &tma_b, &full[stage], kb * BK, n_idx * BN);
          ++issued;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // every load of this CTA is issued: the next kernel may launch
      allow_dependent_launch();
      if (!ok) {
        // let the loads already issued land before the CTA's shared memory
        // can be handed to another CTA (bounded; no abort check)
        volatile int never = 0;
        for (int back = 1; back <= STAGES && back <= issued; ++back) {
          int s = stage - back;
          uint32_t ph = phase;
          if (s < 0) {
            s += STAGES;
            ph ^= 1u;
          }
          mbar_wait_bounded(&full[s], ph, &never);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(BM, BN);
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < num_units && ok; u += gridDim.x) {
        int tile, ks, nks, tt;
        unit_of(u, tile, ks, nks, tt);
        const int kb0 = static_cast<int>(static_cast<int64_t>(ks) * num_k / nks);
        const int kb1 = static_cast<int>(static_cast<int64_t>(ks + 1) * num_k / nks);
        if (!mbar_wait_bounded(&tempty[acc], acc_phase ^ 1u, abort)) {
          record_failure(err, abort, *abort ? DEV_ABORTED : DEV_TIMEOUT_MMA_EMPTY);
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait_spin(&full[stage], phase, abort)) {
            record_failure(err, abort, *abort ? DEV_ABORTED : DEV_TIMEOUT_MMA_FULL);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_addr = smem_u32(sA + stage * A_BYTES);
          const uint32_t b_addr = smem_u32(sB + stage * B_BYTES);
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk)
            umma_bf16(d_tmem, sdesc_k_sw128(a_addr + kk * 32), sdesc_k_sw128(b_addr + kk * 32),
                      idesc, (kb > kb0 || kk > 0) ? 1u : 0u);
          umma_commit(&empty[stage]);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit(&tfull[acc]);
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      if (!ok) {
        // wait (bounded) for every MMA already issued before TMEM is freed
        volatile int never = 0;
        umma_commit(drain);
        mbar_wait_bounded(drain, 0, &never);
      }
    }
  } else {
    const int quad = warp & 3;   // TMEM lane quarter this warp may access
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int u = blockIdx.x; u < num_units; u += gridDim.x) {
      int tile, ks, nks, tt;
      unit_of(u, tile, ks, nks, tt);
      int m_idx, n_idx;
      tile_coords(tile, num_m, num_n, group_m, m_idx, n_idx);
      // a tail unit's fp32 partial: its own BM x BN block of the workspace
      float* tail_ws = tt >= 0 ? ea.ws + (static_cast<int64_t>(tt) * tail_splits + ks) * BM * BN +
                                     static_cast<int64_t>(quad * 32 + lane) * BN
                               : nullptr;
      if (!__all_sync(0xffffffffu, mbar_wait_bounded(&tfull[acc], acc_phase, abort))) {
        if (lane == 0) record_failure(err, abort, *abort ? DEV_ABORTED : DEV_TIMEOUT_EPILOGUE);
        break;
      }
      tc_fence_after();
      const int64_t row = static_cast<int64_t>(m_idx) * BM + quad * 32 + lane;
      const uint32_t t_row = tmem_base + static_cast<uint32_t>(acc * BN) +
                             (static_cast<uint32_t>(quad * 32) << 16);
#pragma unroll 1
      for (int c = 0; c < BN / 32; ++c) {
        const int64_t n0 = static_cast<int64_t>(n_idx) * BN + c * 32;
        if (n0 >= N) break;
        uint32_t r[32];
        tmem_ld_32x32b_x32(t_row + c * 32, r);
        tmem_ld_wait();
        if (row < M) {
          if (tail_ws) {
#pragma unroll
            for (int g = 0; g < 8; ++g)
              *reinterpret_cast<float4*>(tail_ws + c * 32 + 4 * g) =
                  make_float4(__uint_as_float(r[4 * g]), __uint_as_float(r[4 * g + 1]),
                              __uint_as_float(r[4 * g + 2]), __uint_as_float(r[4 * g + 3]));
          } else {
            if (EPI != EPI_PARTIAL && ea.bias) add_bias32(r, ea.bias, n0, N);
            epilogue_store<EPI>(r, row, n0, N, ks, ea);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[acc]);
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

// ---- CTA-pair variant ------------------------------------------------------
//
// A cluster of two CTAs on two SMs computes one 256 x 256 output tile with
// tcgen05.mma.cta_group::2 (M = 256, N = 256, K = 16): CTA r of the pair
// loads rows 128 r .. 128 r + 127 of the tile's A block and of its W block
// (the MMA reads A's rows from both CTAs and the two W halves as one N = 256
// operand) and holds rows 128 r .. of the accumulator in its own tensor
// memory.  Per SM and 64 of K that is 32 KB of operands for the same
// 128 x 256 x 64 products the one-CTA kernel feeds with 48 KB, so more of K
// fits in the ring, and each MMA reads 64 bytes of shared memory per cycle
// instead of 96.
//   warp 0 (both CTAs)  TMA of its halves into its own ring; both signal
//                       the even CTA's `full` barrier, which expects the
//                       bytes of both;
//   warp 1              allocates the pair's tensor memory (with the peer's
//                       warp 1); in the even CTA one thread issues the MMAs,
//                       whose commits arrive on `empty` / `tfull` of both
//                       CTAs;
//   warps 2-5           epilogue of the CTA's 128 rows; they release the
//                       accumulator on the even CTA's `tempty` (8 arrivals).
// A stage holds a k-block of PBK = 128: two 128 x 64 boxes of A and two of W
// per CTA, three stages.  Against 64-wide k-blocks in six stages (the same
// bytes in flight) this halves the MMA thread's barrier waits and commits per
// product, which cost tensor-pipe time: Super's fc1 1.316 -> 1.300 ms, fc2
// 1.322 -> 1.305, the block forward under the power cap 5.73 -> 5.69 ms.
constexpr int BM2 = 256, PBK = 128, PAIR_STAGES = 3;
constexpr int PAIR_A_BOX = (BM2 / 2) * BK * 2;      // 16 KB: 128 rows x 64
constexpr int PAIR_B_BOX = (BN / 2) * BK * 2;       // 16 KB
constexpr int PAIR_A_BYTES = (PBK / BK) * PAIR_A_BOX;
constexpr int PAIR_B_BYTES = (PBK / BK) * PAIR_B_BOX;
constexpr int PAIR_STAGE_BYTES = PAIR_A_BYTES + PAIR_B_BYTES;
constexpr int PAIR_SMEM_BYTES = PAIR_STAGES * PAIR_STAGE_BYTES + 1024 + 256;

// Work units as in the one-CTA kernel without the all-tile split: output
// tiles, then the last `tail` tiles (a short last wave of pairs) as
// `tail_splits` K slices each, whose fp32 partials go to the workspace as
// 256 x 256 blocks for tail_reduce_kernel.
template <int EPI>
__global__ void __launch_bounds__(NUM_THREADS, 1)
gemm_pair_kernel(const __grid_constant__ CUtensorMap tma_a,
                 const __grid_constant__ CUtensorMap tma_b, int M, int N, int K, int tail,
                 int tail_splits, int group_m, const EpiArgs ea, int* err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + PAIR_STAGES * PAIR_A_BYTES;
  uint64_t* full = reinterpret_cast<uint64_t*>(sB + PAIR_STAGES * PAIR_B_BYTES);
  uint64_t* empty = full + PAIR_STAGES;
  uint64_t* tfull = empty + PAIR_STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  constexpr uint16_t kBoth = 0x3;

  if (threadIdx.x == 0) {
    for (int s = 0; s < PAIR_STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 8);
    }
    mbar_init(drain, 1);
    *abort = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tma_a);
    tma_prefetch_desc(&tma_b);
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_slot, TMEM_COLS);
    tmem_relinquish_pair();
  }
  // both CTAs' barriers are initialised before either may signal the other's
  tc_fence_before();
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  grid_dependency_wait();

  const int num_m = (M + BM2 - 1) / BM2;
  const int num_n = (N + BN - 1) / BN;
  const int num_tiles = num_m * num_n;
  const int num_k = (K + PBK - 1) / PBK;
  const int cid = static_cast<int>(cluster_id_x());
  const int ncl = static_cast<int>(cluster_count_x());
  const int n_main = num_tiles - tail;
  const int num_units = n_main + tail * tail_splits;
  // unit -> tile, its k-blocks [kb0, kb1), and (tail units) tail index and slice
  auto unit_of = [&](int u, int& tile, int& kb0, int& kb1, int& tt, int& ks) {
    if (u < n_main) {
      tile = u;
      kb0 = 0;
      kb1 = num_k;
      tt = -1;
      ks = 0;
    } else {
      tt = (u - n_main) / tail_splits;
      ks = (u - n_main) - tt * tail_splits;
      tile = n_main + tt;
      kb0 = static_cast<int>(static_cast<int64_t>(ks) * num_k / tail_splits);
      kb1 = static_cast<int>(static_cast<int64_t>(ks + 1) * num_k / tail_splits);
    }
  };

  if (warp == 0) {
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int u = cid; u < num_units && ok; u += ncl) {
        int t, kb0, kb1, tt, ks;
        unit_of(u, t, kb0, kb1, tt, ks);
        int m_idx, n_idx;
        tile_coords(t, num_m, num_n, group_m, m_idx, n_idx);
        const int arow = m_idx * BM2 + static_cast<int>(rank) * (BM2 / 2);
        const int brow = n_idx * BN + static_cast<int>(rank) * (BN / 2);
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait_spin(&empty[stage], phase ^ 1u, abort)) {
            record_failure(err, abort, *abort ? DEV_ABORTED : DEV_TIMEOUT_PRODUCER);
            ok = false;
            break;
          }
          const uint32_t bar = cluster_addr(&full[stage], 0);
          if (leader) mbar_arrive_expect_tx(&full[stage], 2 * PAIR_STAGE_BYTES);
          for (int h = 0; h < PBK / BK; ++h) {
            tma_load_2d_pair(sA + stage * PAIR_A_BYTES + h * PAIR_A_BOX, &tma_a, bar,
                             kb * PBK + h * BK, arow);
            tma_load_2d_pair(sB + stage * PAIR_B_BYTES + h * PAIR_B_BOX, &tma_b, bar,
                             kb * PBK + h * BK, brow);
          }
          if (++stage == PAIR_STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // every load of this CTA is issued: the next kernel may launch
      allow_dependent_launch();
      if (!ok) {
        // loads already issued signal the even CTA's barriers; give them
        // time to land before the pair can exit (failure path only)
        const uint64_t t0 = globaltimer_ns();
        while (globaltimer_ns() - t0 < 2000000ull) {
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && leader) {
      constexpr uint32_t idesc = idesc_bf16_f32(BM2, BN);
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (int u = cid; u < num_units && ok; u += ncl) {
        int t, kb0, kb1, tt, ks;
        unit_of(u, t, kb0, kb1, tt, ks);
        if (!mbar_wait_spin_cluster(&tempty[acc], acc_phase ^ 1u, abort)) {
          record_failure(err, abort, *abort ? DEV_ABORTED : DEV_TIMEOUT_MMA_EMPTY);
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
        for (int kb = kb0; kb < kb1; ++kb) {
          // (no tcgen05 fence here: the operands were written by TMA, which
          // like the MMA is an async-proxy agent, and the mbarrier's
          // transaction count orders the two)
          if (!mbar_wait_spin(&full[stage], phase, abort)) {
            record_failure(err, abort, *abort ? DEV_ABORTED : DEV_TIMEOUT_MMA_FULL);
            ok = false;
            break;
          }
          const uint32_t a_addr = smem_u32(sA + stage * PAIR_A_BYTES);
          const uint32_t b_addr = smem_u32(sB + stage * PAIR_B_BYTES);
#pragma unroll
          for (int kk = 0; kk < PBK / 16; ++kk)
            umma_bf16_pair(d_tmem,
                           sdesc_k_sw128(a_addr + (kk >> 2) * PAIR_A_BOX + (kk & 3) * 32),
                           sdesc_k_sw128(b_addr + (kk >> 2) * PAIR_B_BOX + (kk & 3) * 32),
                           idesc, (kb > kb0 || kk > 0) ? 1u : 0u);
          umma_commit_pair(&empty[stage], kBoth);
          if (++stage == PAIR_STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit_pair(&tfull[acc], kBoth);
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      // every MMA issued has completed (and its commits have arrived)
      // before either CTA frees tensor memory or exits
      umma_commit_pair(drain, kBoth);
    }
  } else {
    const int quad = warp & 3;
    int acc = 0;
    uint32_t acc_phase = 0;
    const uint32_t tempty_leader0 = cluster_addr(&tempty[0], 0);
    const uint32_t tempty_leader1 = cluster_addr(&tempty[1], 0);
    for (int u = cid; u < num_units; u += ncl) {
      int t, kb0, kb1, tt, ks;
      unit_of(u, t, kb0, kb1, tt, ks);
      int m_idx, n_idx;
      tile_coords(t, num_m, num_n, group_m, m_idx, n_idx);
      const int r_tile = static_cast<int>(rank) * (BM2 / 2) + quad * 32 + lane;  // row in tile
      // a tail unit's fp32 partial: its own BM2 x BN block of the workspace
      float* tail_ws = tt >= 0 ? ea.ws + ((static_cast<int64_t>(tt) * tail_splits + ks) * BM2 +
                                          r_tile) * BN
                               : nullptr;
      if (!__all_sync(0xffffffffu, mbar_wait_bounded(&tfull[acc], acc_phase, abort))) {
        if (lane == 0) record_failure(err, abort, *abort ? DEV_ABORTED : DEV_TIMEOUT_EPILOGUE);
        break;
      }
      tc_fence_after();
      const int64_t row = static_cast<int64_t>(m_idx) * BM2 + r_tile;
      const uint32_t t_row = tmem_base + static_cast<uint32_t>(acc * BN) +
                             (static_cast<uint32_t>(quad * 32) << 16);
#pragma unroll 1
      for (int c = 0; c < BN / 32; ++c) {
        const int64_t n0 = static_cast<int64_t>(n_idx) * BN + c * 32;
        if (n0 >= N) break;
        uint32_t r[32];
        tmem_ld_32x32b_x32(t_row + c * 32, r);
        tmem_ld_wait();
        if (row < M) {
          if (tail_ws) {
#pragma unroll
            for (int g = 0; g < 8; ++g)
              *reinterpret_cast<float4*>(tail_ws + c * 32 + 4 * g) =
                  make_float4(__uint_as_float(r[4 * g]), __uint_as_float(r[4 * g + 1]),
                              __uint_as_float(r[4 * g + 2]), __uint_as_float(r[4 * g + 3]));
          } else {
            if (ea.bias) add_bias32(r, ea.bias, n0, N);
            epilogue_store<EPI>(r, row, n0, N, 0, ea);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(acc == 0 ? tempty_leader0 : tempty_leader1);
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
  }

  // the even CTA's last commit (drain) reaches both CTAs once every MMA of
  // the pair is done; then neither CTA's shared or tensor memory is used by
  // the other any more
  if (warp == 1 && lane == 0) {
    volatile int never = 0;
    if (!mbar_wait_bounded(drain, 0, &never)) record_failure(err, abort, DEV_TIMEOUT_MMA_FULL);
  }
  __syncwarp();
  tc_fence_before();
  cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, TMEM_COLS);
  }
}

int group_rows(int64_t M, int64_t K) {
  const int num_m = static_cast<int>((M + BM - 1) / BM);
  return M * K * 2 <= kAResidentBytes || num_m < kGroupM ? num_m : kGroupM;
}

// The same for the pair kernel's 256-row blocks: groups of 16 of them
// (4,096 rows; a wave of 76 pairs then spans 16 row by ~5 column blocks).
// Measured on one box against 8 and 4 row blocks per group: Super's fc1
// 1.343 / 1.354 / 1.418 ms, Nano's fc2 0.274 / 0.278 / 0.280 ms.
constexpr int kGroupPairM = 16;
int group_rows_pair(int64_t M, int64_t K) {
  const int num_m = static_cast<int>((M + BM2 - 1) / BM2);
  return M * K * 2 <= kAResidentBytes || num_m < kGroupPairM ? num_m : kGroupPairM;
}

template <int EPI>
cudaError_t set_attr() {
  cudaError_t e = cudaFuncSetAttribute(gemm_tcgen05_kernel<EPI>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
  if (e != cudaSuccess || EPI == EPI_PARTIAL) return e;
  return cudaFuncSetAttribute(gemm_pair_kernel<EPI>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              PAIR_SMEM_BYTES);
}

cudaError_t g_attr_err = cudaSuccess;
std::once_flag g_attr_once;
int g_pair_clusters = 0;   // co-resident CTA pairs of the pair kernel (0: not available)

void set_all_attrs() {
  std::call_once(g_attr_once, [] {
    cudaError_t e0 = set_attr<EPI_BF16>(), e1 = set_attr<EPI_GELU_BF16>(),
                e2 = set_attr<EPI_RESID_F32>(), e3 = set_attr<EPI_QKV>(),
                e4 = set_attr<EPI_PARTIAL>();
    const cudaError_t all[5] = {e0, e1, e2, e3, e4};
    g_attr_err = cudaSuccess;
    for (cudaError_t e : all)
      if (e != cudaSuccess) g_attr_err = e;
    if (g_attr_err != cudaSuccess) return;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(2 * sm_count());
    cfg.blockDim = dim3(NUM_THREADS);
    cfg.dynamicSmemBytes = PAIR_SMEM_BYTES;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = 2;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, gemm_pair_kernel<EPI_BF16>, &cfg) != cudaSuccess) {
      cudaGetLastError();
      n = 0;
    }
    g_pair_clusters = n;
  });
}

// -1: choose by shape (pair_auto), 0: never the pair kernel, 1: the pair
// kernel for every linear it can run (tests and measurements).
int g_pair_mode = -1;

// K slices for the tiles of a short last wave of `slots` workers (at least
// 4 k-blocks a slice, at most 8 slices); 1: no split.
int64_t tail_slices(int64_t tiles, int64_t slots, int64_t num_k) {
  const int64_t tail = tiles % slots;
  if (tiles < slots || tail == 0) return 1;
  int64_t ts = slots / tail;
  if (ts > num_k / 4) ts = num_k / 4;
  if (ts > 8) ts = 8;
  return ts >= 2 ? ts : 1;
}

// Estimated time of `tiles` on `slots` workers in k-block steps of a wave:
// fractional waves plus ~40 steps for the reduction when the last wave's
// tiles split, else whole waves.
double wave_cost(int64_t tiles, int64_t slots, int64_t num_k) {
  if (tail_slices(tiles, slots, num_k) > 1)
    return static_cast<double>(tiles) / static_cast<double>(slots) * num_k + 40.0;
  return static_cast<double>((tiles + slots - 1) / slots) * num_k;
}

// The pair kernel runs 256 x 256 tiles in waves of CTA pairs, the one-CTA
// kernel 128 x 256 tiles in waves of SMs; both spread a short last wave over
// the idle workers as K slices, at the cost of a reduction launch.  Both are
// estimated by wave_cost in k-block steps of one wave, the pair kernel's
// steps at 0.9 of the one-CTA kernel's (measured on GB300: 1.86 vs 1.71
// PFLOP/s on Super's fc1).  Grids with fewer pair tiles than pairs keep the
// one-CTA kernel and its K splits of every tile.
bool pair_auto(int64_t M, int64_t N, int64_t K, int clusters) {
  const int64_t tiles2 = ((M + BM2 - 1) / BM2) * ((N + BN - 1) / BN);
  const int64_t num_k = (K + BK - 1) / BK;
  if (tiles2 < clusters || num_k < 4) return false;
  const int64_t tiles1 = ((M + BM - 1) / BM) * ((N + BN - 1) / BN);
  return 0.9 * wave_cost(tiles2, clusters, num_k) < wave_cost(tiles1, sm_count(), num_k);
}

bool use_pair(int64_t M, int64_t N, int64_t K) {
  set_all_attrs();
  if (g_attr_err != cudaSuccess || g_pair_clusters <= 0 || g_pair_mode == 0) return false;
  if (g_pair_mode == 1) return true;
  return pair_auto(M, N, K, g_pair_clusters);
}

template <int EPI>
dlo_status launch_pair(const CUtensorMap& ma, const CUtensorMap& mb, int M, int N, int K,
                       int tail, int tail_splits, const EpiArgs& ea, int* err,
                       cudaStream_t stream) {
  set_all_attrs();
  DLO_CUDA(g_attr_err);
  const int tiles = ((M + BM2 - 1) / BM2) * ((N + BN - 1) / BN);
  const int units = tiles - tail + tail * tail_splits;
  const int clusters = units < g_pair_clusters ? units : g_pair_clusters;
  DLO_CUDA(launch_kernel(gemm_pair_kernel<EPI>, dim3(2 * clusters), dim3(NUM_THREADS),
                         PAIR_SMEM_BYTES, stream, 2, ma, mb, M, N, K, tail, tail_splits,
                         group_rows_pair(M, K), ea, err));
  return DLO_OK;
}


template <int EPI>
dlo_status launch_epi(const CUtensorMap& ma, const CUtensorMap& mb, int M, int N, int K,
                      int splits, int tail, int tail_splits, const EpiArgs& ea, int* err,
                      cudaStream_t stream) {
  set_all_attrs();
  DLO_CUDA(g_attr_err);
  const int tiles = ((M + BM - 1) / BM) * ((N + BN - 1) / BN);
  const int units = (tiles - tail) * splits + tail * tail_splits;
  const int grid = units < sm_count() ? units : sm_count();
  DLO_CUDA(launch_kernel(gemm_tcgen05_kernel<EPI>, dim3(grid), dim3(NUM_THREADS), SMEM_BYTES,
                         stream, 1, ma, mb, M, N, K, splits, tail, tail_splits, group_rows(M, K),
                         ea, err));
  return DLO_OK;
}

// The final epilogue (bf16 store, GELU-tanh, gated residual, or the QKV
// split with V transposed) of four summed outputs at (row, c..c+3).
template <int EPI>
__device__ __forceinline__ void finish4(float4 acc, int64_t row, int64_t c, int64_t N,
                                        const EpiArgs& ea) {
  if (ea.bias) {
    const uint2 b = __ldg(reinterpret_cast<const uint2*>(ea.bias + c));
    acc.x += __uint_as_float(b.x << 16);
    acc.y += __uint_as_float(b.x & 0xFFFF0000u);
    acc.z += __uint_as_float(b.y << 16);
    acc.w += __uint_as_float(b.y & 0xFFFF0000u);
  }
  if (EPI == EPI_QKV && c >= ea.v_col0) {
    // V columns (v_col0 is a multiple of 64, so all four are V): vt[b*d + c', t]
    const int64_t b = row / ea.tokens, t = row - b * ea.tokens;
    const int64_t d = ea.v_col0 / 2;
    uint16_t* dst = ea.vt + (b * d + (c - ea.v_col0)) * ea.vt_ld + t;
    const float v[4] = {acc.x, acc.y, acc.z, acc.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      __nv_bfloat16 h = __float2bfloat16_rn(v[i]);
      dst[static_cast<int64_t>(i) * ea.vt_ld] = *reinterpret_cast<uint16_t*>(&h);
    }
    return;
  }
  if (EPI == EPI_RESID_F32) {
    float4* xp = reinterpret_cast<float4*>(static_cast<float*>(ea.out) + row * N + c);
    const float4 gv = __ldg(reinterpret_cast<const float4*>(ea.gate + c));
    float4 xv = *xp;
    xv.x += gv.x * acc.x;
    xv.y += gv.y * acc.y;
    xv.z += gv.z * acc.z;
    xv.w += gv.w * acc.w;
    *xp = xv;
  } else {
    if (EPI == EPI_GELU_BF16) {
      acc.x = gelu_tanh(acc.x);
      acc.y = gelu_tanh(acc.y);
      acc.z = gelu_tanh(acc.z);
      acc.w = gelu_tanh(acc.w);
    }
    __nv_bfloat162 p0 = __floats2bfloat162_rn(acc.x, acc.y);
    __nv_bfloat162 p1 = __floats2bfloat162_rn(acc.z, acc.w);
    uint2 pk;
    pk.x = *reinterpret_cast<uint32_t*>(&p0);
    pk.y = *reinterpret_cast<uint32_t*>(&p1);
    *reinterpret_cast<uint2*>(static_cast<uint16_t*>(ea.out) + row * N + c) = pk;
  }
}

__device__ __forceinline__ void add4(float4& acc, const float* p) {
  const float4 v = *reinterpret_cast<const float4*>(p);
  acc.x += v.x;
  acc.y += v.y;
  acc.z += v.z;
  acc.w += v.w;
}

// Sums the K slices of a split linear, ws [splits, M, N], in slice order and
// applies the final epilogue.
template <int EPI>
__global__ void __launch_bounds__(256)
splitk_reduce_kernel(const float* __restrict__ ws, int splits, int64_t M, int64_t N,
                     const EpiArgs ea) {
  grid_dependency_sync();
  const int64_t n4 = N / 4, total = M * n4;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t row = i / n4, c = (i - row * n4) * 4;
    float4 acc = *reinterpret_cast<const float4*>(ws + row * N + c);
    for (int s = 1; s < splits; ++s) add4(acc, ws + (s * M + row) * N + c);
    finish4<EPI>(acc, row, c, N, ea);
  }
}

// The same for the tail tiles only: ws [tail, tail_splits, TM, BN], tail
// tile tt being output tile num_tiles - tail + tt (tile t at row block
// and column block from tile_coords); TM = BM for the one-CTA kernel's
// tiles, BM2 for the pair kernel's.
template <int EPI, int TM>
__global__ void __launch_bounds__(256)
tail_reduce_kernel(const float* __restrict__ ws, int tail, int tail_splits, int num_tiles,
                   int num_m, int num_n, int group_m, int64_t M, int64_t N,
                   const EpiArgs ea) {
  grid_dependency_sync();
  constexpr int64_t per_tile = static_cast<int64_t>(TM) * (BN / 4);
  const int64_t total = tail * per_tile;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int tt = static_cast<int>(i / per_tile);
    const int64_t e = i - tt * per_tile;
    const int64_t r = e / (BN / 4), c = (e - r * (BN / 4)) * 4;
    const int tile = num_tiles - tail + tt;
    int m_idx, n_idx;
    tile_coords(tile, num_m, num_n, group_m, m_idx, n_idx);
    const int64_t row = static_cast<int64_t>(m_idx) * TM + r;
    const int64_t col = static_cast<int64_t>(n_idx) * BN + c;
    if (row >= M || col >= N) continue;
    const float* p = ws + (static_cast<int64_t>(tt) * tail_splits * TM + r) * BN + c;
    float4 acc = *reinterpret_cast<const float4*>(p);
    for (int s = 1; s < tail_splits; ++s) add4(acc, p + static_cast<int64_t>(s) * TM * BN);
    finish4<EPI>(acc, row, col, N, ea);
  }
}

template <int EPI, int TM = BM>
dlo_status launch_tail_reduce(const float* ws, int tail, int tail_splits, int64_t M, int64_t N,
                              int64_t K, const EpiArgs& ea, cudaStream_t stream) {
  const int num_m = static_cast<int>((M + TM - 1) / TM);
  const int num_n = static_cast<int>((N + BN - 1) / BN);
  const int num_tiles = num_m * num_n;
  const int64_t total = static_cast<int64_t>(tail) * TM * (BN / 4);
  int64_t blocks = (total + 255) / 256;
  const int64_t cap = static_cast<int64_t>(sm_count()) * 8;
  if (blocks > cap) blocks = cap;
  const int group_m = TM == BM ? group_rows(M, K) : group_rows_pair(M, K);
  DLO_CUDA(launch_kernel(tail_reduce_kernel<EPI, TM>, dim3(static_cast<unsigned>(blocks)),
                         dim3(256), 0, stream, 1, ws, tail, tail_splits, num_tiles, num_m,
                         num_n, group_m, M, N, ea));
  return DLO_OK;
}

template <int EPI>
dlo_status launch_reduce(const float* ws, int splits, int64_t M, int64_t N, const EpiArgs& ea,
                         cudaStream_t stream) {
  const int64_t total = M * (N / 4);
  int64_t blocks = (total + 255) / 256;
  const int64_t cap = static_cast<int64_t>(sm_count()) * 8;
  if (blocks > cap) blocks = cap;
  DLO_CUDA(launch_kernel(splitk_reduce_kernel<EPI>, dim3(static_cast<unsigned>(blocks)),
                         dim3(256), 0, stream, 1, ws, splits, M, N, ea));
  return DLO_OK;
}

// The pair kernel, then (a split tail) the ordered reduction of its tail
// tiles' K slices with the epilogue.
template <int EPI>
dlo_status launch_pair_linear(const CUtensorMap& ma, const CUtensorMap& mb, int M, int N, int K,
                              int tail, int tail_splits, const EpiArgs& ea, int* err,
                              cudaStream_t stream) {
  DLO_TRY(launch_pair<EPI>(ma, mb, M, N, K, tail, tail_splits, ea, err, stream));
  if (tail == 0) return DLO_OK;
  return launch_tail_reduce<EPI, BM2>(ea.ws, tail, tail_splits, M, N, K, ea, stream);
}

}  // namespace

LinearPlan linear_plan(int64_t M, int64_t N, int64_t K, int epilogue) {
  LinearPlan p{1, 0, 1, 0, 1, 0};
  if (epilogue != EPI_PARTIAL && use_pair(M, N, K)) {
    p.pair = 1;
    const int64_t tiles2 = ((M + BM2 - 1) / BM2) * ((N + BN - 1) / BN);
    const int64_t ts = tail_slices(tiles2, g_pair_clusters, (K + BK - 1) / BK);
    if (ts > 1) {
      p.tail = static_cast<int>(tiles2 % g_pair_clusters);
      p.tail_splits = static_cast<int>(ts);
      p.ws_bytes = static_cast<size_t>(p.tail) * ts * BM2 * BN * 4;
      p.launches = 2;
    }
    return p;
  }
  const int64_t sms = sm_count();
  const int64_t tiles = ((M + BM - 1) / BM) * ((N + BN - 1) / BN);
  const int64_t num_k = (K + BK - 1) / BK;
  auto clamp = [&](int64_t s) {
    if (s > num_k / 4) s = num_k / 4;    // every slice keeps at least 4 k-blocks
    if (s > 8) s = 8;
    return s;
  };
  // fewer tiles than SMs: every tile split
  const int64_t s = clamp(sms / (tiles > 0 ? tiles : 1));
  if (s >= 2) {
    p.splits = static_cast<int>(s);
    p.ws_bytes = static_cast<size_t>(s) * M * N * 4;
    p.launches = 2;
    return p;
  }
  // a last wave of at most half the SMs: its tiles split over the idle SMs
  const int64_t tail = tiles % sms;
  if (tiles >= sms && tail > 0) {
    const int64_t ts = clamp(sms / tail);
    if (ts >= 2) {
      p.tail = static_cast<int>(tail);
      p.tail_splits = static_cast<int>(ts);
      p.ws_bytes = static_cast<size_t>(tail) * ts * BM * BN * 4;
      p.launches = 2;
    }
  }
  return p;
}

int linear_splits(int64_t M, int64_t N, int64_t K, int epilogue) {
  return linear_plan(M, N, K, epilogue).splits;
}

size_t linear_workspace_bytes(int64_t M, int64_t N, int64_t K, int epilogue) {
  return linear_plan(M, N, K, epilogue).ws_bytes;
}

namespace {
}  // namespace

dlo_status set_gemm_pair_mode(int mode) {
  if (mode < -1 || mode > 1) DLO_FAIL(DLO_ERR_INVALID, "gemm pair mode %d (expected -1, 0, 1)", mode);
  g_pair_mode = mode;
  return DLO_OK;
}

int gemm_pair_mode() { return g_pair_mode; }

dlo_status gemm_preload() {
  set_all_attrs();
  DLO_CUDA(g_attr_err);
  sm_count();
  return DLO_OK;
}

dlo_status launch_linear_ex(const uint16_t* a, int64_t M, int64_t K, const uint16_t* w,
                            int64_t N, int epilogue, const EpiArgs& ea, cudaStream_t stream) {
  if (M == 0) return DLO_OK;
  if (!a || !w || !ea.out || M < 0 || K <= 0 || N <= 0)
    DLO_FAIL(DLO_ERR_INVALID, "linear: bad arguments (M %lld, K %lld, N %lld)", (long long)M,
             (long long)K, (long long)N);
  if (K % 8 != 0 || N % 8 != 0)
    DLO_FAIL(DLO_ERR_INVALID, "linear: K (%lld) and N (%lld) must be multiples of 8",
             (long long)K, (long long)N);
  if (M > (1LL << 31) - 1 || N > (1LL << 31) - 1 || K > (1LL << 31) - 1)
    DLO_FAIL(DLO_ERR_INVALID, "linear: extent too large");
  if ((reinterpret_cast<uintptr_t>(a) | reinterpret_cast<uintptr_t>(w) |
       reinterpret_cast<uintptr_t>(ea.out)) & 15u)
    DLO_FAIL(DLO_ERR_INVALID, "linear: a, w and out must be 16-byte aligned");
  if (ea.bias && (reinterpret_cast<uintptr_t>(ea.bias) & 15u))
    DLO_FAIL(DLO_ERR_INVALID, "linear: the bias must be 16-byte aligned");
  if (epilogue == EPI_RESID_F32 && (!ea.gate || (reinterpret_cast<uintptr_t>(ea.gate) & 15u)))
    DLO_FAIL(DLO_ERR_INVALID, "linear: the residual epilogue needs a 16-byte aligned gate");
  if (epilogue == EPI_QKV &&
      (!ea.vt || ea.tokens <= 0 || ea.v_col0 <= 0 || ea.v_col0 % 64 != 0 || ea.vt_ld < ea.tokens ||
       N != ea.v_col0 / 2 * 3))
    DLO_FAIL(DLO_ERR_INVALID, "linear: bad arguments for the QKV epilogue");
  int* err = device_error_word();
  if (!err) DLO_FAIL(DLO_ERR_CUDA, "linear: cannot resolve the device error word");
  const int m = static_cast<int>(M), n = static_cast<int>(N), k = static_cast<int>(K);
  const LinearPlan plan = linear_plan(M, N, K, epilogue);
  CUtensorMap ma, mb;
  if (plan.pair) {
    DLO_TRY(make_tmap_2d(&ma, a, M, K, K, BM2 / 2, BK));
    DLO_TRY(make_tmap_2d(&mb, w, N, K, K, BN / 2, BK));
    // the tail's K slices need the workspace; without it the tail runs whole
    const bool split = plan.tail > 0 && ea.ws && ea.ws_bytes >= plan.ws_bytes &&
                       !(reinterpret_cast<uintptr_t>(ea.ws) & 15u);
    const int tl = split ? plan.tail : 0, ts = split ? plan.tail_splits : 1;
    switch (epilogue) {
      case EPI_BF16: return launch_pair_linear<EPI_BF16>(ma, mb, m, n, k, tl, ts, ea, err, stream);
      case EPI_GELU_BF16:
        return launch_pair_linear<EPI_GELU_BF16>(ma, mb, m, n, k, tl, ts, ea, err, stream);
      case EPI_RESID_F32:
        return launch_pair_linear<EPI_RESID_F32>(ma, mb, m, n, k, tl, ts, ea, err, stream);
      case EPI_QKV: return launch_pair_linear<EPI_QKV>(ma, mb, m, n, k, tl, ts, ea, err, stream);
      default: DLO_FAIL(DLO_ERR_INVALID, "linear: unknown epilogue %d", epilogue);
    }
  }
  DLO_TRY(make_tmap_2d(&ma, a, M, K, K, BM, BK));
  DLO_TRY(make_tmap_2d(&mb, w, N, K, K, BN, BK));
  const bool have_ws = plan.ws_bytes > 0 && ea.ws && ea.ws_bytes >= plan.ws_bytes &&
                       !(reinterpret_cast<uintptr_t>(ea.ws) & 15u);
  const int splits = plan.splits;
  if (splits > 1 && have_ws) {
    // K split across CTAs: fp32 partials, then an ordered reduction with
    // the epilogue (deterministic: the slice order is fixed)
    EpiArgs pa = ea;
    pa.ws_rows = M;
    DLO_TRY(launch_epi<EPI_PARTIAL>(ma, mb, m, n, k, splits, 0, 1, pa, err, stream));
    switch (epilogue) {
      case EPI_BF16: return launch_reduce<EPI_BF16>(ea.ws, splits, M, N, ea, stream);
      case EPI_GELU_BF16: return launch_reduce<EPI_GELU_BF16>(ea.ws, splits, M, N, ea, stream);
      case EPI_RESID_F32: return launch_reduce<EPI_RESID_F32>(ea.ws, splits, M, N, ea, stream);
      case EPI_QKV: return launch_reduce<EPI_QKV>(ea.ws, splits, M, N, ea, stream);
      default: DLO_FAIL(DLO_ERR_INVALID, "linear: unknown epilogue %d", epilogue);
    }
  }
  if (plan.tail > 0 && have_ws) {
    // the short last wave's tiles split in K (partials in ws), the others
    // finished in the kernel; then the tail's ordered reduction
    const int tl = plan.tail, ts = plan.tail_splits;
    switch (epilogue) {
      case EPI_BF16:
        DLO_TRY(launch_epi<EPI_BF16>(ma, mb, m, n, k, 1, tl, ts, ea, err, stream));
        return launch_tail_reduce<EPI_BF16>(ea.ws, tl, ts, M, N, K, ea, stream);
      case EPI_GELU_BF16:
        DLO_TRY(launch_epi<EPI_GELU_BF16>(ma, mb, m, n, k, 1, tl, ts, ea, err, stream));
        return launch_tail_reduce<EPI_GELU_BF16>(ea.ws, tl, ts, M, N, K, ea, stream);
      case EPI_RESID_F32:
        DLO_TRY(launch_epi<EPI_RESID_F32>(ma, mb, m, n, k, 1, tl, ts, ea, err, stream));
        return launch_tail_reduce<EPI_RESID_F32>(ea.ws, tl, ts, M, N, K, ea, stream);
      case EPI_QKV:
        DLO_TRY(launch_epi<EPI_QKV>(ma, mb, m, n, k, 1, tl, ts, ea, err, stream));
        return launch_tail_reduce<EPI_QKV>(ea.ws, tl, ts, M, N, K, ea, stream);
      default: DLO_FAIL(DLO_ERR_INVALID, "linear: unknown epilogue %d", epilogue);
    }
  }
  switch (epilogue) {
    case EPI_BF16: return launch_epi<EPI_BF16>(ma, mb, m, n, k, 1, 0, 1, ea, err, stream);
    case EPI_GELU_BF16:
      return launch_epi<EPI_GELU_BF16>(ma, mb, m, n, k, 1, 0, 1, ea, err, stream);
    case EPI_RESID_F32:
      return launch_epi<EPI_RESID_F32>(ma, mb, m, n, k, 1, 0, 1, ea, err, stream);
    case EPI_QKV: return launch_epi<EPI_QKV>(ma, mb, m, n, k, 1, 0, 1, ea, err, stream);
    default: DLO_FAIL(DLO_ERR_INVALID, "linear: unknown epilogue %d", epilogue);
  }
}

dlo_status launch_linear(const uint16_t* a, int64_t M, int64_t K, const uint16_t* w, int64_t N,
                         int epilogue, void* out, const float* gate, const uint16_t* bias,
                         float* ws, size_t ws_bytes, cudaStream_t stream) {
  if (epilogue == EPI_QKV) DLO_FAIL(DLO_ERR_INVALID, "linear: the QKV epilogue is internal");
  EpiArgs ea{};
  ea.out = out;
  ea.gate = gate;
  ea.bias = bias;
  ea.ws = ws;
  ea.ws_bytes = ws_bytes;
  return launch_linear_ex(a, M, K, w, N, epilogue, ea, stream);
}

}  // namespace dlo
