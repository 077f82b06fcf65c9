// common.h — internal helpers shared by the library's translation units:
// status/error reporting, CUDA checks, the plan's in-memory form and the
// launchers each kernel file exports to the host-side orchestration.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdio>
#include <string>
#include <utility>
#include <vector>

#include "../../include/dlo.h"

namespace dlo {

// Thread-local message behind dlo_last_error().
void set_error(const char* fmt, ...);
void clear_error();

#define DLO_FAIL(code, ...)          \
  do {                               \
    ::dlo::set_error(__VA_ARGS__);   \
    return (code);                   \
  } while (0)

#define DLO_CUDA(call)                                                     \
  do {                                                                     \
    cudaError_t err_ = (call);                                             \
    if (err_ != cudaSuccess)                                               \
      DLO_FAIL(DLO_ERR_CUDA, "%s failed: %s (%s:%d)", #call,               \
               cudaGetErrorString(err_), __FILE__, __LINE__);              \
  } while (0)

#define DLO_TRY(expr)                         \
  do {                                        \
    dlo_status st_ = (expr);                  \
    if (st_ != DLO_OK) return st_;            \
  } while (0)

constexpr int64_t kGroupAlign = 256;
constexpr int kMaxSegments = 64;   // (dtype group, shard) pairs per prefetch

inline int64_t round_up(int64_t v, int64_t a) { return (v + a - 1) / a * a; }

// Roles of the synthetic DiT block's parameters: the first R_REQUIRED are
// required; the rest are the checkpoint-shaped block's optional ones (bf16
// biases of the four linears, fp32 per-head q/k RMSNorm gains).
enum Role {
  R_G1 = 0, R_SHIFT1, R_SCALE1, R_GATE1, R_WQKV, R_WO,
  R_G2, R_SHIFT2, R_SCALE2, R_GATE2, R_W1, R_W2, R_REQUIRED,
  R_BQKV = R_REQUIRED, R_BO, R_B1, R_B2, R_QNORM, R_KNORM, R_COUNT
};
extern const char* const kRoleNames[R_COUNT];

}  // namespace dlo

struct dlo_plan {
  struct Param {
    std::string name;
    int32_t ndim;
    int64_t shape[4];
    int32_t dtype;
    int64_t numel;          // logical elements
    int64_t stride[4];      // element strides of the view (row-major if contiguous)
    bool contiguous;
    int64_t storage_numel;  // elements packed: the view's storage extent
    int32_t group;
    int64_t group_offset;   // elements
    int64_t slot_offset;    // bytes
  };
  struct Group {
    int32_t dtype;
    int32_t esize;
    int64_t numel;
    int64_t shard_numel;
    int64_t shard_bytes;
    int64_t shard_alloc_bytes;
    int64_t base;
    int64_t stage_base;     // first shard's offset in a staging buffer
  };
  std::vector<Param> params;
  std::vector<Group> groups;
  int32_t n_shards = 1;
  int64_t slot_bytes = 0;
  int64_t staging_bytes = 0;
  int32_t role[dlo::R_COUNT];   // param index per role, -1 if absent
  bool has_dit_roles = false;
  uint64_t id = 0;              // unique per plan (keys cached graphs)
};

namespace dlo {

// One host->device piece of a prefetch: a shard and its final place.
struct Segment {
  const void* src;    // device-accessible address of the pinned host shard
  void* dst;          // slot + base_g + r * shard_bytes
  int64_t bytes;      // shard_bytes
};

struct SegmentTable {
  int32_t n;
  Segment seg[kMaxSegments];
};

// copy_kernel.cu
dlo_status launch_copy_reassemble(const SegmentTable& t, int ctas,
                                  cudaStream_t stream);

// norm.cu
dlo_status launch_rmsnorm_mod(const float* x, int64_t rows, int64_t d,
                              const float* g, const float* shift,
                              const float* scale, float eps, uint16_t* h,
                              cudaStream_t stream);

// gemm.cu
// EPI_QKV: columns [0, 2d) stored bf16 like EPI_BF16, columns [2d, 3d)
// (the V block) stored transposed into vt[b*d + c, t] (row stride vt_ld).
// EPI_PARTIAL (internal): fp32 partial sums of one K slice into ws.
enum Epilogue {
  EPI_BF16 = 0, EPI_GELU_BF16 = 1, EPI_RESID_F32 = 2, EPI_QKV = 3, EPI_PARTIAL = 4
};
struct EpiArgs {
  void* out;            // bf16 [M, N], or fp32 x [M, N] for the residual
  const float* gate;    // [N], residual epilogue
  uint16_t* vt;         // EPI_QKV: V transposed
  int64_t vt_ld;        // EPI_QKV: row stride of vt (>= tokens)
  int tokens;           // EPI_QKV: rows per batch item
  int v_col0;           // EPI_QKV: first V column (2d)
  const uint16_t* bias; // bf16 [N] added to the product before the epilogue (null: none)
  float* ws;            // split-K workspace [splits, M, N] fp32 (null: no split)
  size_t ws_bytes;
  int64_t ws_rows;      // M, set for the partial epilogue
};
// How a linear of this shape is run on this GPU's SMs: on CTA pairs in
// 256 x 256 tiles (`pair`, when the tiles fill the pairs' waves well), else
// on single CTAs with `splits` K slices
// for every tile (fewer tiles than SMs), or `tail_splits` K slices for the
// last `tail` tiles only (a last wave of at most half the SMs); the fp32
// workspace that needs and the kernel launches (2 with a reduction).
// Without a large enough workspace a linear runs unsplit.
struct LinearPlan {
  int splits;
  int tail;
  int tail_splits;
  size_t ws_bytes;
  int launches;
  int pair;             // 1: unsplit on CTA pairs (gemm_pair_kernel), 256 x 256 tiles
};
LinearPlan linear_plan(int64_t M, int64_t N, int64_t K, int epilogue);
int linear_splits(int64_t M, int64_t N, int64_t K, int epilogue);
size_t linear_workspace_bytes(int64_t M, int64_t N, int64_t K, int epilogue);
dlo_status launch_linear(const uint16_t* a, int64_t M, int64_t K,
                         const uint16_t* w, int64_t N, int epilogue, void* out,
                         const float* gate, const uint16_t* bias, float* ws, size_t ws_bytes,
                         cudaStream_t stream);
// Per-head RMSNorm (gains gq, gk [hd]; both null: none) and rotary
// embedding (rope_base > 0; 0: none) of the q and k columns of the bf16 qkv
// buffer [batch*tokens, 3d], in place.
dlo_status launch_qk_norm_rope(uint16_t* qkv, int64_t batch, int64_t tokens, int64_t d,
                               int64_t heads, const float* gq, const float* gk, float eps,
                               float rope_base, cudaStream_t stream);
dlo_status launch_linear_ex(const uint16_t* a, int64_t M, int64_t K, const uint16_t* w,
                            int64_t N, int epilogue, const EpiArgs& ea, cudaStream_t stream);

// attention.cu
int64_t vt_ld_for(int64_t tokens);   // row stride of vt: tokens rounded up to 8
// How attention runs on this GPU's SMs: nt query tiles per CTA, `items`
// (batch, head, query group) items of which the first n_main run whole and
// the rest (a last wave of at most half the SMs) as `parts` KV slices each,
// merged by a second kernel; `units` CTAs, the fp32 workspace of the slices
// and the launches (1, or 2 with the merge).
struct AttPlan {
  int nt;
  int64_t items, n_main, units;
  int parts;
  size_t ws_bytes;
  int launches;
};
AttPlan attention_plan(int64_t batch, int64_t tokens, int64_t d, int64_t heads);
// ws: the slices' workspace (ws_bytes >= attention_plan(...).ws_bytes), or
// null: then every item runs whole.
dlo_status launch_attention_vt(const uint16_t* qkv, const uint16_t* vt, int64_t vt_ld,
                               int64_t batch, int64_t tokens, int64_t d, int64_t heads,
                               uint16_t* o, float* ws, size_t ws_bytes, cudaStream_t stream);
dlo_status launch_transpose_v(const uint16_t* qkv, int64_t batch, int64_t tokens, int64_t d,
                              uint16_t* vt, int64_t vt_ld, cudaStream_t stream);

// tmap.cu: TMA descriptors and device facts
// Row-major bf16 matrix [rows, cols] with a row stride of `ld` elements as
// TMA boxes of box_rows x box_cols (box_cols * 2 = 128 bytes with the
// 128-byte swizzle); out-of-range elements read as zero.
dlo_status make_tmap_2d(CUtensorMap* map, const void* ptr, int64_t rows, int64_t cols,
                        int64_t ld, uint32_t box_rows, uint32_t box_cols);
int sm_count();

// Launches of the block forward: inside a PdlScope(true) (this thread),
// kernels are launched with programmatic stream serialization, so that a
// kernel's CTAs may start their set-up while the previous kernel drains
// (each waits for it in grid_dependency_wait/sync before touching memory).
// cluster_x > 1 launches clusters of that many CTAs.
bool pdl_active();
struct PdlScope {
  bool prev;
  explicit PdlScope(bool on);
  ~PdlScope();
};
int launch_overlap_mode();   // -1 by block size (default), 0 off, 1 on

template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                          cudaStream_t stream, int cluster_x, Args&&... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute at[2];
  unsigned n = 0;
  if (cluster_x > 1) {
    at[n].id = cudaLaunchAttributeClusterDimension;
    at[n].val.clusterDim.x = static_cast<unsigned>(cluster_x);
    at[n].val.clusterDim.y = 1;
    at[n].val.clusterDim.z = 1;
    ++n;
  }
  if (pdl_active()) {
    at[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  cfg.attrs = at;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// status.cu: device-side error word written by bounded waits
int* device_error_word();  // device address (cached per device)

// One-time per-process preparation of each kernel (function attributes,
// module loading), so that no first-launch cost lands in a timed window or
// inside a graph capture.
dlo_status gemm_preload();
dlo_status set_gemm_pair_mode(int mode);   // -1 by shape, 0 never, 1 always
int gemm_pair_mode();
dlo_status attention_preload();
dlo_status copy_preload();

}  // namespace dlo
