// attention.cu — non-causal softmax attention of the synthetic DiT block on
// the 5th-generation tensor cores.
//
// o[b, t, head j] = softmax_u( q_t . k_u / sqrt(hd) ) v_u per batch item and
// head.  Q and K are the first two hd-wide column blocks of head j in the
// bf16 qkv buffer [batch*tokens, 3d]; V is read transposed, vt[b*d + j*hd +
// c, u] (keys contiguous), which the QKV linear's epilogue writes directly,
// so that both products below take K-major operands.
//
// One CTA = two 128-query tiles (Q_0, Q_1) of one (batch, head) that share
// every K and V tile: KV tiles of 128 keys stream once through shared memory
// for 256 queries.  (Grids that would then have fewer CTAs than SMs run one
// query tile per CTA instead; WG1 then idles.)  Three warpgroups:
//   WG0, WG1   softmax of Q_0 and Q_1, one thread per query row (its TMEM
//              lane); each finally writes its tile of o;
//   WG2        warp 8: TMA of the two Q tiles, then K_0, V_0, K_1, V_1, ...
//              into one NS-stage ring (NS = 5 for hd 128, 12 for hd 64);
//              warp 9: TMEM allocation (512 columns) and the tcgen05.mma
//              issue.
// WG2 gives up registers to the softmax warpgroups (setmaxnreg), which hold
// a whole row of scores.
// TMEM: S_t at column 128 t (fp32, 128 keys); P_t (bf16, two per column)
// overwrites the first 64 columns of S_t; O_t at column 256 + hd t.
// MMA order: S_0(0) S_1(0), then per KV tile j
//   PV_0(j)  O_0 += P_0(j) V_j   (A = P_0 from TMEM, B = V_j^T in smem)
//   S_0(j+1) = Q_0 K_{j+1}^T     (after PV_0(j) in issue order, so P_0(j)
//                                 is read before S_0(j+1) overwrites it)
//   PV_1(j), S_1(j+1).
// While softmax t turns S_t(j+1) into P_t(j+1) the tensor pipe runs the
// other tile's PV and S.  The commit that signals S_t(j+1) also covers
// PV_t(j), so softmax t may then rescale O_t and overwrite P_t.
// The MMA thread keeps its own synchronisation to one wait, one fence and
// one commit per query tile and KV tile (each costs tensor-pipe time, the
// issue queue being shallow): it waits only for P_t(j); the softmax warps
// check that V_j and K_{j+1} have landed before they signal P, and the last
// query tile's softmax releases the ring stages (its S commit covers every
// earlier product).
// Softmax per tile: the 128 scores of the row with one TMEM load wait; the
// first KV tile fixes m (its row maximum); later ones keep it unless a row's
// sum of P over the tile reaches kGrowSum, which moves m up to the row's
// maximum, rescales O_t and l and recomputes the tile's P; P =
// 2^(s*scale - m) as bf16 into TMEM with tcgen05.st, row sum l.  At the end
// o = O_t / l.  Keys past the end are -inf in S and zero in V (TMA zero
// fill).  All waits are bounded; a wait that runs out records a code in the
// device error word and the kernel returns early.
#include <cuda_bf16.h>

#include <mutex>

#include "common.h"
#include "ptx.cuh"

namespace dlo {
namespace {

constexpr int BQ = 128, BKV = 128, ATT_THREADS = 384;
constexpr uint32_t ATT_TMEM_COLS = 512;
// A query tile keeps the row maximum m of its first KV tile until a row's
// sum of P over one KV tile reaches this (2^64): every P of a kept tile is
// then below 2^64, far from the fp32 and bf16 range limits (without loss of
// relative precision), and O needs no rescaling in the common case.
constexpr float kGrowSum = 18446744073709551616.f;

template <int HD>
struct AttLayout {
  static constexpr int NS = HD == 128 ? 5 : 12;        // K/V ring stages
  static constexpr int Q_TILE = BQ * HD * 2;           // HD/64 chunks of 128 rows x 128 B
  static constexpr int K_CHUNK = BKV * 128;            // 128 keys x 64 dims
  static constexpr int V_CHUNK = HD * 128;             // HD rows x 64 keys
  static constexpr int KV_BYTES = BKV * HD * 2;        // one K or V^T tile
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_KV = OFF_Q + 2 * Q_TILE;
  static constexpr int OFF_BAR = OFF_KV + NS * KV_BYTES;
  static constexpr int SMEM = OFF_BAR + 512 + 1024;    // barriers + alignment slack
};

// Register budget per thread after the split (setmaxnreg): the issue
// warpgroup gives up what the two softmax warpgroups take, so the total stays
// the launch's 384 x 168.
constexpr int kRegsLaunch = 168, kRegsIssue = 120, kRegsSoftmax = 192;
static_assert(kRegsIssue * 128 + kRegsSoftmax * 256 == kRegsLaunch * ATT_THREADS,
              "register split must add up to the launch's registers");

template <int N>
__device__ __forceinline__ void reg_dealloc() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}
template <int N>
__device__ __forceinline__ void reg_alloc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}

__device__ __forceinline__ void att_fail(int* err, volatile int* abort, int code) {
  atomicCAS(err, 0, *abort ? static_cast<int>(DEV_ABORTED) : code);
  *abort = 1;
}

// 2^x by the hardware approximation (MUFU.EX2 through the PTX instruction;
// denormal results flush to zero, 2^-inf = 0).
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&p);
}

// Packed pairs of fp32 (Blackwell's paired FMA/add pipes): lane 0 in the
// low 32 bits.
__device__ __forceinline__ uint64_t f2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ float f2_lo(uint64_t v) { return __uint_as_float(static_cast<uint32_t>(v)); }
__device__ __forceinline__ float f2_hi(uint64_t v) {
  return __uint_as_float(static_cast<uint32_t>(v >> 32));
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}

// 32 lanes x 128 consecutive columns in one instruction (thread l: row lane
// base + l); valid after tmem_ld_wait().
__device__ __forceinline__ void tmem_ld_32x32b_x128(uint32_t taddr, uint32_t (&r)[128]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x128.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63,%64,%65,%66,%67,%68,%69,%70,%71,%72,%73,%74,%75,%76,%77,%78,%79,%80,%81,%82,%83,%84,%85,%86,%87,%88,%89,%90,%91,%92,%93,%94,%95,%96,%97,%98,%99,%100,%101,%102,%103,%104,%105,%106,%107,%108,%109,%110,%111,%112,%113,%114,%115,%116,%117,%118,%119,%120,%121,%122,%123,%124,%125,%126,%127}, [%128];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63]), "=r"(r[64]), "=r"(r[65]), "=r"(r[66]), "=r"(r[67]), "=r"(r[68]), "=r"(r[69]), "=r"(r[70]), "=r"(r[71]), "=r"(r[72]), "=r"(r[73]), "=r"(r[74]), "=r"(r[75]), "=r"(r[76]), "=r"(r[77]), "=r"(r[78]), "=r"(r[79]), "=r"(r[80]), "=r"(r[81]), "=r"(r[82]), "=r"(r[83]), "=r"(r[84]), "=r"(r[85]), "=r"(r[86]), "=r"(r[87]), "=r"(r[88]), "=r"(r[89]), "=r"(r[90]), "=r"(r[91]), "=r"(r[92]), "=r"(r[93]), "=r"(r[94]), "=r"(r[95]), "=r"(r[96]), "=r"(r[97]), "=r"(r[98]), "=r"(r[99]), "=r"(r[100]), "=r"(r[101]), "=r"(r[102]), "=r"(r[103]), "=r"(r[104]), "=r"(r[105]), "=r"(r[106]), "=r"(r[107]), "=r"(r[108]), "=r"(r[109]), "=r"(r[110]), "=r"(r[111]), "=r"(r[112]), "=r"(r[113]), "=r"(r[114]), "=r"(r[115]), "=r"(r[116]), "=r"(r[117]), "=r"(r[118]), "=r"(r[119]), "=r"(r[120]), "=r"(r[121]), "=r"(r[122]), "=r"(r[123]), "=r"(r[124]), "=r"(r[125]), "=r"(r[126]), "=r"(r[127])
               : "r"(taddr)
               : "memory");
}

// Inverse of the load above for 64 columns.
__device__ __forceinline__ void tmem_st_32x32b_x64(uint32_t taddr, const uint32_t (&r)[64]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x64.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63,%64};"
               :
               : "r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31]), "r"(r[32]), "r"(r[33]), "r"(r[34]), "r"(r[35]), "r"(r[36]), "r"(r[37]), "r"(r[38]), "r"(r[39]), "r"(r[40]), "r"(r[41]), "r"(r[42]), "r"(r[43]), "r"(r[44]), "r"(r[45]), "r"(r[46]), "r"(r[47]), "r"(r[48]), "r"(r[49]), "r"(r[50]), "r"(r[51]), "r"(r[52]), "r"(r[53]), "r"(r[54]), "r"(r[55]), "r"(r[56]), "r"(r[57]), "r"(r[58]), "r"(r[59]), "r"(r[60]), "r"(r[61]), "r"(r[62]), "r"(r[63])
               : "memory");
}

__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// The 128 fp32 scores of this thread's row (TMEM lane) from taddr: one
// load, one wait.  Scores of keys at or past `valid` become -inf.
__device__ __forceinline__ void load_row(uint32_t taddr, int valid, uint32_t (&sr)[BKV]) {
  tmem_ld_32x32b_x128(taddr, sr);
  tmem_ld_wait();
  if (valid < BKV) {
#pragma unroll
    for (int i = 0; i < BKV; ++i)
      if (i >= valid) sr[i] = __float_as_uint(-INFINITY);
  }
}

// Maximum of a row's 128 scores (-inf if all are).
__device__ __forceinline__ float row_max(const uint32_t (&sr)[BKV]) {
  float mx[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) mx[e] = __uint_as_float(sr[e]);
#pragma unroll
  for (int i = 4; i < BKV; i += 8)
#pragma unroll
    for (int e = 0; e < 4; ++e)
      mx[e] = fmax3(mx[e], __uint_as_float(sr[i + e]),
                    i + 4 + e < BKV ? __uint_as_float(sr[i + 4 + e]) : -INFINITY);
  return fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
}

// P = 2^(s * scale - m) for a row's 128 scores, as 64 bf16 pairs written
// over sr[0..63] (pair h from scores 2h, 2h+1, which no later pair reads);
// returns the row sum of P (fp32, before the bf16 rounding), accumulated in
// four packed pairs of partial sums.
__device__ __forceinline__ float exp_row(uint32_t (&sr)[BKV], float m, float scale_log2) {
  const uint64_t sc2 = f2(scale_log2, scale_log2), nm2 = f2(-m, -m);
  uint64_t ls[4] = {0, 0, 0, 0};
#pragma unroll
  for (int h = 0; h < BKV / 2; ++h) {
    const uint64_t x = f2_fma(f2(__uint_as_float(sr[2 * h]), __uint_as_float(sr[2 * h + 1])),
                              sc2, nm2);
    const uint64_t pp = f2(ex2_approx(f2_lo(x)), ex2_approx(f2_hi(x)));
    ls[h & 3] = f2_add(ls[h & 3], pp);
    sr[h] = pack_bf16(f2_lo(pp), f2_hi(pp));
  }
  const uint64_t l2 = f2_add(f2_add(ls[0], ls[1]), f2_add(ls[2], ls[3]));
  return f2_lo(l2) + f2_hi(l2);
}

// Multiplies this warp's 32 lanes x (32 * CHUNKS) fp32 columns from taddr by
// each lane's corr.
template <int CHUNKS>
__device__ __forceinline__ void rescale_tmem_f32(uint32_t taddr, float corr) {
#pragma unroll 1
  for (int c = 0; c < CHUNKS; ++c) {
    uint32_t r[32];
    tmem_ld_32x32b_x32(taddr + c * 32, r);
    tmem_ld_wait();
#pragma unroll
    for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * corr);
    tmem_st_32x32b_x32(taddr + c * 32, r);
  }
}

// Four back-to-back kind::f16 products into one accumulator, both operands
// in shared memory (descriptors a[i], b[i]); the first accumulates only if
// acc != 0, the other three always.  One asm block, so that no other
// instruction of the issuing thread sits between the products: the tensor
// pipe's issue queue is shallow, and each instruction between two products
// is tensor time lost.
__device__ __forceinline__ void umma_ss_x4(uint32_t d, const uint64_t (&a)[4],
                                           const uint64_t (&b)[4], uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.b32 p, %9, 0;\n\t"
      "setp.eq.b32 q, %9, %9;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %5, %10, p;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %2, %6, %10, q;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %3, %7, %10, q;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %4, %8, %10, q;\n\t}" ::"r"(d),
      "l"(a[0]), "l"(a[1]), "l"(a[2]), "l"(a[3]), "l"(b[0]), "l"(b[1]), "l"(b[2]), "l"(b[3]),
      "r"(acc), "r"(idesc)
      : "memory");
}

// The same with the A operands in tensor memory (column addresses ta[i]).
__device__ __forceinline__ void umma_ts_x4(uint32_t d, const uint32_t (&ta)[4],
                                           const uint64_t (&b)[4], uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.b32 p, %9, 0;\n\t"
      "setp.eq.b32 q, %9, %9;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %5, %10, p;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%2], %6, %10, q;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%3], %7, %10, q;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%4], %8, %10, q;\n\t}" ::"r"(d),
      "r"(ta[0]), "r"(ta[1]), "r"(ta[2]), "r"(ta[3]), "l"(b[0]), "l"(b[1]), "l"(b[2]), "l"(b[3]),
      "r"(acc), "r"(idesc)
      : "memory");
}

template <int HD>
__global__ void __launch_bounds__(ATT_THREADS, 1)
attention_tc_kernel(const __grid_constant__ CUtensorMap tm_qk,
                    const __grid_constant__ CUtensorMap tm_vt, int tokens, int d, int heads,
                    uint16_t* __restrict__ o, float scale_log2, int nt, int n_main, int parts,
                    float* __restrict__ part_ws, int* err) {
  using L = AttLayout<HD>;
  constexpr int NS = L::NS;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = smem + L::OFF_Q;
  uint8_t* sKV = smem + L::OFF_KV;
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + L::OFF_BAR);
  uint64_t* q_full = bar;
  uint64_t* full = bar + 1;                  // [NS]
  uint64_t* empty = full + NS;               // [NS]
  uint64_t* s_full = empty + NS;             // [2]  per query tile
  uint64_t* p_full = s_full + 2;             // [2]
  uint64_t* o_done = p_full + 2;             // [2]
  uint64_t* drain = o_done + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int wg = warp >> 2;
  // Unit blockIdx.x: the first n_main are whole (batch, head, query group)
  // items (nt query tiles), numbered query group fastest, then head, then
  // batch; each later one is a slice `part` of the KV tiles of one of the
  // remaining items (a short last wave spread over the idle SMs), which
  // writes its unnormalised O, m and l to part_ws for attention_combine.
  const int n_groups = (tokens + nt * BQ - 1) / (nt * BQ);
  const int u = blockIdx.x;
  const int item = u < n_main ? u : n_main + (u - n_main) / parts;
  const int part = u < n_main ? -1 : (u - n_main) % parts;
  const int q0 = (item % n_groups) * nt * BQ;
  const int head = (item / n_groups) % heads, b = item / (n_groups * heads);
  const int n_kv_all = (tokens + BKV - 1) / BKV;
  const int kv_base = part < 0 ? 0 : part * n_kv_all / parts;
  // KV tiles of this unit: kv_base .. kv_base + n_kv - 1 (local index j)
  const int n_kv = part < 0 ? n_kv_all : (part + 1) * n_kv_all / parts - kv_base;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&s_full[t], 1);
      mbar_init(&p_full[t], 4);
      mbar_init(&o_done[t], 1);
    }
    mbar_init(drain, 1);
    *abort = 0;
    fence_mbar_init();
  }
  if (warp == 8 && lane == 0) {
    tma_prefetch_desc(&tm_qk);
    tma_prefetch_desc(&tm_vt);
  }
  if (warp == 9) {
    tmem_alloc(tmem_slot, ATT_TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  grid_dependency_sync();
  const uint32_t tS = tmem;             // S_t (and P_t) at column 128 t
  const uint32_t tO = tmem + 256;       // O_t at column 256 + HD t

  if (wg == 2) {
    // the loader and MMA issuer need few registers; the softmax warpgroups
    // take them (launch 384 x 168 = 128 x 120 + 256 x 192)
    reg_dealloc<kRegsIssue>();
    if (warp == 8 && lane == 0) {
      // load i = 2j is K_j, i = 2j+1 is V_j; stage i % NS, use i / NS
      mbar_arrive_expect_tx(q_full, nt * L::Q_TILE);
      for (int t = 0; t < nt; ++t)
        for (int c = 0; c < HD / 64; ++c)
          tma_load_2d(sQ + t * L::Q_TILE + c * (BQ * 128), &tm_qk, q_full, head * HD + 64 * c,
                      b * tokens + q0 + t * BQ);
      int issued = 0;
      for (int i = 0; i < 2 * n_kv; ++i) {
        const int s = i % NS;
        const uint32_t use = static_cast<uint32_t>(i / NS);
        const int kv0 = (kv_base + (i >> 1)) * BKV;
        if (!mbar_wait_bounded(&empty[s], (use & 1u) ^ 1u, abort)) {
          att_fail(err, abort, DEV_TIMEOUT_PRODUCER);
          break;
        }
        mbar_arrive_expect_tx(&full[s], L::KV_BYTES);
        uint8_t* dst = sKV + s * L::KV_BYTES;
        if ((i & 1) == 0) {
          for (int c = 0; c < HD / 64; ++c)
            tma_load_2d(dst + c * L::K_CHUNK, &tm_qk, &full[s], d + head * HD + 64 * c,
                        b * tokens + kv0);
        } else {
          for (int c = 0; c < 2; ++c)
            tma_load_2d(dst + c * L::V_CHUNK, &tm_vt, &full[s], kv0 + 64 * c,
                        (b * heads + head) * HD);
        }
        ++issued;
      }
      if (*abort) {
        // let the copies already issued land before the CTA can exit
        volatile int never = 0;
        mbar_wait_bounded(q_full, 0, &never);
        for (int i = issued - NS < 0 ? 0 : issued - NS; i < issued; ++i)
          mbar_wait_bounded(&full[i % NS], static_cast<uint32_t>((i / NS) & 1), &never);
      }
    } else if (warp == 9 && lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16_f32(BQ, BKV);
      constexpr uint32_t idesc_o = idesc_bf16_f32(BQ, HD);
      // Each tcgen05.mma occupies the issuing thread for about as long as
      // the tensor pipe needs to execute it, so everything between two MMAs
      // costs tensor time: descriptors are formed once and advanced by
      // constant offsets (the 14-bit start-address field never carries, as
      // shared-memory addresses are below 256 KB), and the groups are fully
      // unrolled.
      const uint64_t dq = sdesc_k_sw128(smem_u32(sQ));
      const uint64_t dkv = sdesc_k_sw128(smem_u32(sKV));
      auto wait_load = [&](int i) {
        return mbar_wait_spin(&full[i % NS], static_cast<uint32_t>((i / NS) & 1), abort);
      };
      // S_t = Q_t K^T with K in stage s, in groups of four products
      auto mma_s = [&](int t, int s) {
        const uint64_t a = dq + static_cast<uint64_t>((t * L::Q_TILE) >> 4);
        const uint64_t b = dkv + static_cast<uint64_t>((s * L::KV_BYTES) >> 4);
#pragma unroll
        for (int g = 0; g < HD / 64; ++g) {
          uint64_t ad[4], bd[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            ad[e] = a + static_cast<uint64_t>((g * (BQ * 128) + e * 32) >> 4);
            bd[e] = b + static_cast<uint64_t>((g * L::K_CHUNK + e * 32) >> 4);
          }
          umma_ss_x4(tS + t * BKV, ad, bd, idesc_s, g > 0 ? 1u : 0u);
        }
      };
      // O_t += P_t V with V^T in stage s
      auto mma_pv = [&](int t, int s, bool acc) {
        const uint64_t b = dkv + static_cast<uint64_t>((s * L::KV_BYTES) >> 4);
#pragma unroll
        for (int g = 0; g < BKV / 64; ++g) {
          uint32_t ta[4];
          uint64_t bd[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            ta[e] = tS + t * BKV + (4 * g + e) * 8;
            bd[e] = b + static_cast<uint64_t>((g * L::V_CHUNK + e * 32) >> 4);
          }
          umma_ts_x4(tO + t * HD, ta, bd, idesc_o, g > 0 || acc ? 1u : 0u);
        }
      };
      bool ok = mbar_wait_bounded(q_full, 0, abort) && wait_load(0);
      if (ok) {
        tc_fence_after();
        mma_s(0, 0);
        umma_commit(&s_full[0]);
        if (nt == 2) {
          mma_s(1, 0);
          umma_commit(&s_full[1]);
        }
      }
      // The MMA thread's own barrier reads, fences and commits cost
      // tensor-pipe time (the issue queue is shallow), so it keeps one of
      // each per query tile and KV tile: it waits only for P_t(j), whose
      // softmax warps have first checked that V_j and K_{j+1} landed, and
      // commits only the S_t(j+1) (or final O_t) signal; the softmax of the
      // last query tile releases the K/V stages.
      int sv = 1 % NS, sk = 2 % NS;              // stages of V_j and K_{j+1}
      for (int j = 0; ok && j < n_kv; ++j) {
        const uint32_t par = static_cast<uint32_t>(j & 1);
        const bool more = j + 1 < n_kv;
        if (!mbar_wait_spin(&p_full[0], par, abort)) {
          ok = false;
          break;
        }
        tc_fence_after();
        mma_pv(0, sv, j > 0);
        if (more) {
          mma_s(0, sk);
          umma_commit(&s_full[0]);
        } else {
          umma_commit(&o_done[0]);
        }
        if (nt == 2) {
          if (!mbar_wait_spin(&p_full[1], par, abort)) {
            ok = false;
            break;
          }
          tc_fence_after();
          mma_pv(1, sv, j > 0);
          if (more) {
            mma_s(1, sk);
            umma_commit(&s_full[1]);
          } else {
            umma_commit(&o_done[1]);
          }
        }
        sv = sv + 2 >= NS ? sv + 2 - NS : sv + 2;
        sk = sk + 2 >= NS ? sk + 2 - NS : sk + 2;
      }
      if (!ok) {
        att_fail(err, abort, DEV_TIMEOUT_MMA_FULL);
        volatile int never = 0;
        umma_commit(drain);
        mbar_wait_bounded(drain, 0, &never);
      }
    }
  } else if (wg < nt) {
    reg_alloc<kRegsSoftmax>();
    const int t = wg;                          // query tile of this warpgroup
    const int quad = warp & 3;
    const int row = quad * 32 + lane;          // query row in the tile == TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const uint32_t tSt = tS + t * BKV + lane_off, tOt = tO + t * HD + lane_off;
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < n_kv; ++j) {
      if (!__all_sync(0xffffffffu,
                      mbar_wait_bounded(&s_full[t], static_cast<uint32_t>(j & 1), abort))) {
        if (lane == 0) att_fail(err, abort, DEV_TIMEOUT_EPILOGUE);
        ok = false;
        break;
      }
      tc_fence_after();
      // S_t(j) complete: for the last query tile this commit also covers
      // PV(j-1) and S(j) of every tile, so the stages of V_{j-1} and K_j are
      // free for the loader
      if (t == nt - 1 && quad == 0 && lane == 0) {
        if (j > 0) mbar_arrive(&empty[(2 * j - 1) % NS]);
        mbar_arrive(&empty[(2 * j) % NS]);
      }
      // PV_t(j) reads V_j and S_t(j+1) reads K_{j+1}: one thread of the
      // warpgroup sees both loads complete before the warpgroup signals P
      // (tested now, waited for only if not yet complete at the end)
      const int iv = 2 * j + 1, ik = 2 * j + 2;
      const bool more = j + 1 < n_kv;
      const bool chk = quad == 0 && lane == 0;
      bool loads_ok = true;
      if (chk) {
        const bool v_ok = mbar_test(&full[iv % NS], static_cast<uint32_t>((iv / NS) & 1));
        const bool k_ok = !more || mbar_test(&full[ik % NS], static_cast<uint32_t>((ik / NS) & 1));
        loads_ok = v_ok && k_ok;
      }
      const int valid = tokens - (kv_base + j) * BKV;   // keys of this tile that exist
      // the whole row of S_t at once: one TMEM load wait per KV tile
      uint32_t sr[BKV];
      load_row(tSt, valid, sr);
      if (j == 0) m = row_max(sr) * scale_log2;   // the first KV tile fixes m
      // P = exp2(s * scale - m) as bf16 pairs, then its row sum
      float lt = exp_row(sr, m, scale_log2);
      // A row whose scores outgrew m (its P sum reached kGrowSum, or is not
      // finite) moves m up to its maximum and redoes the tile: O_t (PV_t(j-1)
      // has completed: it precedes S_t(j) in issue order) and l are scaled
      // by 2^(m_old - m_new) and P is recomputed from S_t, still in TMEM.
      if (__any_sync(0xffffffffu, !(lt < kGrowSum))) {
        const bool need = !(lt < kGrowSum);
        float cm = -INFINITY;                 // the row maximum, 32 scores at a time
#pragma unroll 1
        for (int c = 0; c < BKV / 32; ++c) {
          uint32_t r[32];
          tmem_ld_32x32b_x32(tSt + c * 32, r);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 32; ++i)
            if (32 * c + i < valid) cm = fmaxf(cm, __uint_as_float(r[i]));
        }
        cm *= scale_log2;
        float corr = 1.f;
        if (need && cm > m) {
          corr = ex2_approx(m - cm);
          m = cm;
        }
        l *= corr;
        rescale_tmem_f32<HD / 32>(tOt, corr);
        load_row(tSt, valid, sr);
        lt = exp_row(sr, m, scale_log2);
      }
      // P over the first 64 columns of S_t
      tmem_st_32x32b_x64(tSt, *reinterpret_cast<const uint32_t(*)[64]>(&sr[0]));
      l += lt;
      if (chk && !loads_ok) {
        loads_ok = mbar_wait_bounded(&full[iv % NS], static_cast<uint32_t>((iv / NS) & 1), abort) &&
                   (!more ||
                    mbar_wait_bounded(&full[ik % NS], static_cast<uint32_t>((ik / NS) & 1), abort));
        if (!loads_ok) att_fail(err, abort, DEV_TIMEOUT_ATTN);
      }
      tmem_st_wait();
      tc_fence_before();
      if (!__all_sync(0xffffffffu, loads_ok)) {
        ok = false;
        break;
      }
      if (lane == 0) mbar_arrive(&p_full[t]);
    }
    if (ok && !__all_sync(0xffffffffu, mbar_wait_bounded(&o_done[t], 0, abort))) {
      if (lane == 0) att_fail(err, abort, DEV_TIMEOUT_EPILOGUE);
      ok = false;
    }
    if (ok && !*abort && part >= 0) {
      // a KV slice: O (fp32, not yet divided by l), then m and l, per row
      tc_fence_after();
      const int64_t slot = (static_cast<int64_t>(item - n_main) * parts + part) * nt + t;
      float* orow = part_ws + (slot * BQ + row) * HD;
#pragma unroll 1
      for (int c = 0; c < HD / 32; ++c) {
        uint32_t oa[32];
        tmem_ld_32x32b_x32(tOt + c * 32, oa);
        tmem_ld_wait();
#pragma unroll
        for (int g = 0; g < 8; ++g)
          *reinterpret_cast<float4*>(orow + c * 32 + 4 * g) =
              make_float4(__uint_as_float(oa[4 * g]), __uint_as_float(oa[4 * g + 1]),
                          __uint_as_float(oa[4 * g + 2]), __uint_as_float(oa[4 * g + 3]));
      }
      const int64_t n_slots = static_cast<int64_t>(gridDim.x - n_main) * nt;
      *reinterpret_cast<float2*>(part_ws + n_slots * BQ * HD + (slot * BQ + row) * 2) =
          make_float2(m, l);
    } else if (ok && !*abort) {
      tc_fence_after();
      const float inv = 1.f / l;
      const int q = q0 + t * BQ + row;
      uint16_t* orow = o + (static_cast<int64_t>(b) * tokens + q) * d + head * HD;
#pragma unroll 1
      for (int c = 0; c < HD / 32; ++c) {
        uint32_t oa[32];
        tmem_ld_32x32b_x32(tOt + c * 32, oa);
        tmem_ld_wait();
        if (q < tokens) {
#pragma unroll
          for (int g = 0; g < 4; ++g) {
            float v[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) v[e] = __uint_as_float(oa[8 * g + e]) * inv;
            *reinterpret_cast<uint4*>(orow + c * 32 + 8 * g) =
                make_uint4(pack_bf16(v[0], v[1]), pack_bf16(v[2], v[3]), pack_bf16(v[4], v[5]),
                           pack_bf16(v[6], v[7]));
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, ATT_TMEM_COLS);
  }
}

// Merges the KV slices of the split items: for each of their query rows,
// M = max_p m_p, o = sum_p 2^(m_p - M) O_p / sum_p 2^(m_p - M) l_p, the
// parts taken in order.  One warp per row, HD / 32 columns per lane.
template <int HD>
__global__ void __launch_bounds__(256)
attention_combine_kernel(const float* __restrict__ part_ws, int n_main, int n_split, int parts,
                         int nt, int tokens, int d, int heads, uint16_t* __restrict__ o) {
  constexpr int CPL = HD / 32;                      // columns per lane
  grid_dependency_sync();
  const int64_t w = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  const int64_t rows = static_cast<int64_t>(n_split) * nt * BQ;
  if (w >= rows) return;
  const int si = static_cast<int>(w / (nt * BQ));   // split item
  const int t = static_cast<int>((w / BQ) % nt), row = static_cast<int>(w % BQ);
  const int item = n_main + si;
  const int n_groups = (tokens + nt * BQ - 1) / (nt * BQ);
  const int q = (item % n_groups) * nt * BQ + t * BQ + row;
  if (q >= tokens) return;
  const int head = (item / n_groups) % heads, b = item / (n_groups * heads);
  const int64_t n_slots = static_cast<int64_t>(n_split) * parts * nt;
  const float* ml = part_ws + n_slots * BQ * HD;
  float mx = -INFINITY;
  for (int p = 0; p < parts; ++p) {
    const int64_t slot = (static_cast<int64_t>(si) * parts + p) * nt + t;
    mx = fmaxf(mx, ml[(slot * BQ + row) * 2]);
  }
  float acc[CPL], l = 0.f;
#pragma unroll
  for (int c = 0; c < CPL; ++c) acc[c] = 0.f;
  for (int p = 0; p < parts; ++p) {
    const int64_t slot = (static_cast<int64_t>(si) * parts + p) * nt + t;
    const float wgt = exp2f(ml[(slot * BQ + row) * 2] - mx);
    l += wgt * ml[(slot * BQ + row) * 2 + 1];
    const float* op = part_ws + (slot * BQ + row) * HD + lane * CPL;
#pragma unroll
    for (int c = 0; c < CPL; ++c) acc[c] += wgt * op[c];
  }
  const float inv = 1.f / l;
  uint16_t* orow = o + (static_cast<int64_t>(b) * tokens + q) * d + head * HD + lane * CPL;
#pragma unroll
  for (int c = 0; c < CPL; c += 2)
    *reinterpret_cast<uint32_t*>(orow + c) = pack_bf16(acc[c] * inv, acc[c + 1] * inv);
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
int g_att_regs[2] = {0, 0};          // registers per thread of <64>, <128>
std::once_flag g_att_once;

void set_att_attrs() {
  std::call_once(g_att_once, [] {
    cudaError_t e0 = cudaFuncSetAttribute(attention_tc_kernel<64>,
                                          cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          AttLayout<64>::SMEM);
    cudaError_t e1 = cudaFuncSetAttribute(attention_tc_kernel<128>,
                                          cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          AttLayout<128>::SMEM);
    cudaFuncAttributes a64{}, a128{};
    cudaError_t e2 = cudaFuncGetAttributes(&a64, attention_tc_kernel<64>);
    cudaError_t e3 = cudaFuncGetAttributes(&a128, attention_tc_kernel<128>);
    g_att_regs[0] = a64.numRegs;
    g_att_regs[1] = a128.numRegs;
    g_att_err = e0 != cudaSuccess ? e0 : e1 != cudaSuccess ? e1 : e2 != cudaSuccess ? e2 : e3;
  });
}

// The register split inside the kernel (setmaxnreg) redistributes exactly
// the registers the CTA is launched with; a build that gave the kernel any
// other count would leave the softmax warpgroups waiting for registers that
// do not exist, so it is refused before launch.
dlo_status check_att_attrs() {
  set_att_attrs();
  DLO_CUDA(g_att_err);
  if (g_att_regs[0] != kRegsLaunch || g_att_regs[1] != kRegsLaunch)
    DLO_FAIL(DLO_ERR_CUDA, "attention: kernel built with %d / %d registers per thread, the "
             "register split needs %d", g_att_regs[0], g_att_regs[1], kRegsLaunch);
  return DLO_OK;
}

template <int HD>
dlo_status launch_hd(const CUtensorMap& tm_qk, const CUtensorMap& tm_vt, const AttPlan& pl,
                     int64_t tokens, int64_t d, int64_t heads, uint16_t* o, float* ws, int* err,
                     cudaStream_t stream) {
  DLO_TRY(check_att_attrs());
  const float scale_log2 = 1.4426950408889634f / sqrtf(static_cast<float>(HD));
  const int n_split = static_cast<int>(pl.items - pl.n_main);
  DLO_CUDA(launch_kernel(attention_tc_kernel<HD>, dim3(static_cast<unsigned>(pl.units)),
                         dim3(ATT_THREADS), AttLayout<HD>::SMEM, stream, 1, tm_qk, tm_vt,
                         static_cast<int>(tokens), static_cast<int>(d), static_cast<int>(heads),
                         o, scale_log2, pl.nt, static_cast<int>(pl.n_main), pl.parts, ws, err));
  if (n_split > 0) {
    const int64_t rows = static_cast<int64_t>(n_split) * pl.nt * BQ;
    DLO_CUDA(launch_kernel(attention_combine_kernel<HD>,
                           dim3(static_cast<unsigned>((rows * 32 + 255) / 256)), dim3(256), 0,
                           stream, 1, static_cast<const float*>(ws),
                           static_cast<int>(pl.n_main), n_split, pl.parts, pl.nt,
                           static_cast<int>(tokens), static_cast<int>(d),
                           static_cast<int>(heads), o));
  }
  return DLO_OK;
}

}  // namespace

int64_t vt_ld_for(int64_t tokens) { return (tokens + 7) / 8 * 8; }

AttPlan attention_plan(int64_t batch, int64_t tokens, int64_t d, int64_t heads) {
  AttPlan p{};
  p.nt = 1;
  p.parts = 1;
  p.launches = 1;
  if (batch <= 0 || tokens <= 0 || heads <= 0 || d % heads != 0) return p;
  const int64_t hd = d / heads;
  const int64_t sms = sm_count();
  // Two query tiles per CTA halve the K/V traffic per query; when that
  // leaves SMs idle (fewer CTAs than SMs), one tile per CTA doubles the CTAs.
  const int64_t pairs = (tokens + 2 * BQ - 1) / (2 * BQ);
  p.nt = pairs * heads * batch >= sms ? 2 : 1;
  p.items = (tokens + p.nt * BQ - 1) / (p.nt * BQ) * heads * batch;
  p.n_main = p.items;
  p.units = p.items;
  // a last wave of at most half the SMs: its items' KV tiles are split over
  // the idle SMs (at least 2 KV tiles per slice)
  const int64_t tail = p.items % sms, n_kv = (tokens + BKV - 1) / BKV;
  if (p.items >= sms && tail > 0) {
    int64_t parts = sms / tail;
    if (parts > n_kv / 2) parts = n_kv / 2;
    if (parts >= 2) {
      p.parts = static_cast<int>(parts);
      p.n_main = p.items - tail;
      p.units = p.n_main + tail * parts;
      p.ws_bytes = static_cast<size_t>(tail) * parts * p.nt * BQ * (hd + 2) * 4;
      p.launches = 2;
    }
  }
  return p;
}

dlo_status attention_preload() { return check_att_attrs(); }

dlo_status launch_attention_vt(const uint16_t* qkv, const uint16_t* vt, int64_t vt_ld,
                               int64_t batch, int64_t tokens, int64_t d, int64_t heads,
                               uint16_t* o, float* ws, size_t ws_bytes, cudaStream_t stream) {
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
  AttPlan pl = attention_plan(batch, tokens, d, heads);
  if (pl.parts > 1 && (!ws || ws_bytes < pl.ws_bytes || (reinterpret_cast<uintptr_t>(ws) & 15u))) {
    // no room for the KV slices: the tail runs whole
    pl.parts = 1;
    pl.n_main = pl.units = pl.items;
  }
  if (pl.units > 0x7fffffffLL) DLO_FAIL(DLO_ERR_INVALID, "attention: too many work units");
  if (hd == 64) return launch_hd<64>(tm_qk, tm_vt, pl, tokens, d, heads, o, ws, err, stream);
  return launch_hd<128>(tm_qk, tm_vt, pl, tokens, d, heads, o, ws, err, stream);
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
