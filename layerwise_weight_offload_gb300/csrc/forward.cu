// forward.cu — the synthetic DiT block forward over weights laid out as a
// slot, and the single-step entry points used by the per-kernel checks.
//
// The pages run the block forward on a compute stream that waits for the
// gather event ("Distributed Layerwise Offload" (vLLM blog preview,
// 2026-07-30), "Weight Sharding + AllGather", step 4) with parameters
// re-pointed into the gathered buffer (step 3).  Here the re-pointing is the
// plan's slot offsets added to the slot's base; the forward is one stream
// of launches:
//   rmsnorm_mod -> linear(qkv, bf16; V transposed) [-> q/k norm + rotary
//   embedding] -> attention -> linear(out, gated residual) -> rmsnorm_mod ->
//   linear(fc1, GELU) -> linear(fc2, gated residual),
// each linear followed by its ordered reduction when some of its tiles run
// as K slices, and attention by the merge of its KV slices.
#include <algorithm>
#include <mutex>
#include <utility>

#include "common.h"
#include "trace.h"

namespace dlo {
namespace {

// Rotary embedding base of the checkpoint-shaped block (DLO_FWD_ROPE): the
// RoFormer value.
constexpr float kRopeBase = 10000.f;

struct ScratchLayout {
  size_t h, qkv, vt, o, u, ws, ws_bytes, total;
  int64_t vt_ld;
};

// Scratch of one forward: bf16 h [M, d] (both norms), qkv [M, 3d] (Q and K
// used), vt [batch*d, vt_ld] (V transposed), o [M, d], u [M, f], and the
// fp32 K-slice workspace of the linear that needs the most (0 if none
// splits; one buffer serves all four, as they run one after the other).
ScratchLayout scratch_layout(const dlo_dit_cfg& c) {
  const size_t M = static_cast<size_t>(c.batch) * c.tokens;
  const size_t d = c.hidden, f = c.mlp;
  auto r = [](size_t v) { return (v + 255) / 256 * 256; };
  ScratchLayout s;
  s.vt_ld = vt_ld_for(c.tokens);
  s.h = 0;
  s.qkv = r(s.h + M * d * 2);
  s.vt = r(s.qkv + M * 3 * d * 2);
  s.o = r(s.vt + static_cast<size_t>(c.batch) * d * static_cast<size_t>(s.vt_ld) * 2);
  s.u = r(s.o + M * d * 2);
  s.ws = r(s.u + M * f * 2);
  const int64_t Mi = static_cast<int64_t>(M), di = c.hidden, fi = c.mlp;
  size_t w = linear_workspace_bytes(Mi, 3 * di, di, EPI_QKV);
  w = std::max(w, attention_plan(c.batch, c.tokens, c.hidden, c.heads).ws_bytes);
  w = std::max(w, linear_workspace_bytes(Mi, di, di, EPI_RESID_F32));
  w = std::max(w, linear_workspace_bytes(Mi, fi, di, EPI_GELU_BF16));
  w = std::max(w, linear_workspace_bytes(Mi, di, fi, EPI_RESID_F32));
  s.ws_bytes = w;
  s.total = r(s.ws + w);
  return s;
}

dlo_status check_cfg(const dlo_dit_cfg* c) {
  if (!c) DLO_FAIL(DLO_ERR_INVALID, "forward: null config");
  if (c->batch < 1 || c->tokens < 1 || c->hidden < 64 || c->heads < 1 || c->mlp < 64)
    DLO_FAIL(DLO_ERR_INVALID, "forward: batch/tokens/hidden/heads/mlp out of range");
  if (c->hidden % 64 != 0 || c->mlp % 64 != 0)
    DLO_FAIL(DLO_ERR_INVALID, "forward: hidden (%d) and mlp (%d) must be multiples of 64",
             c->hidden, c->mlp);
  if (c->hidden % c->heads != 0 ||
      (c->hidden / c->heads != 64 && c->hidden / c->heads != 128))
    DLO_FAIL(DLO_ERR_INVALID, "forward: head dim %d x %d not supported (64 or 128)",
             c->hidden, c->heads);
  if (!(c->eps >= 0.f)) DLO_FAIL(DLO_ERR_INVALID, "forward: eps must be >= 0");
  return DLO_OK;
}

dlo_status check_plan(const dlo_dit_cfg& c, const dlo_plan* plan) {
  if (!plan) DLO_FAIL(DLO_ERR_INVALID, "forward: null plan");
  if (!plan->has_dit_roles)
    DLO_FAIL(DLO_ERR_INVALID, "forward: the plan's parameter names are not the DiT block's");
  const int64_t d = c.hidden, f = c.mlp;
  struct Want { int role; int32_t dtype; int64_t a, b; };
  const Want want[] = {
      {R_G1, DLO_F32, d, 0},      {R_SHIFT1, DLO_F32, d, 0}, {R_SCALE1, DLO_F32, d, 0},
      {R_GATE1, DLO_F32, d, 0},   {R_WQKV, DLO_BF16, 3 * d, d}, {R_WO, DLO_BF16, d, d},
      {R_G2, DLO_F32, d, 0},      {R_SHIFT2, DLO_F32, d, 0}, {R_SCALE2, DLO_F32, d, 0},
      {R_GATE2, DLO_F32, d, 0},   {R_W1, DLO_BF16, f, d},    {R_W2, DLO_BF16, d, f}};
  for (const Want& w : want) {
    const auto& p = plan->params[plan->role[w.role]];
    const bool ok = p.dtype == w.dtype &&
                    (w.b == 0 ? (p.ndim == 1 && p.shape[0] == w.a)
                              : (p.ndim == 2 && p.shape[0] == w.a && p.shape[1] == w.b));
    if (!ok) DLO_FAIL(DLO_ERR_INVALID, "forward: parameter %s has the wrong shape or dtype",
                      kRoleNames[w.role]);
    if (p.slot_offset % 16 != 0)
      DLO_FAIL(DLO_ERR_INVALID, "forward: parameter %s is not 16-byte aligned in the slot",
               kRoleNames[w.role]);
  }
  // the checkpoint-shaped block's optional parameters: biases used when
  // present; q/k norm gains exactly when the configuration asks for them
  const int64_t hd = d / c.heads;
  const Want opt[] = {{R_BQKV, DLO_BF16, 3 * d, 0}, {R_BO, DLO_BF16, d, 0},
                      {R_B1, DLO_BF16, f, 0},       {R_B2, DLO_BF16, d, 0},
                      {R_QNORM, DLO_F32, hd, 0},    {R_KNORM, DLO_F32, hd, 0}};
  for (const Want& w : opt) {
    if (plan->role[w.role] < 0) continue;
    const auto& p = plan->params[plan->role[w.role]];
    if (p.dtype != w.dtype || p.ndim != 1 || p.shape[0] != w.a)
      DLO_FAIL(DLO_ERR_INVALID, "forward: parameter %s has the wrong shape or dtype",
               kRoleNames[w.role]);
    if (p.slot_offset % 16 != 0)
      DLO_FAIL(DLO_ERR_INVALID, "forward: parameter %s is not 16-byte aligned in the slot",
               kRoleNames[w.role]);
  }
  const bool has_qk = plan->role[R_QNORM] >= 0 && plan->role[R_KNORM] >= 0;
  const bool want_qk = (c.flags & DLO_FWD_QK_NORM) != 0;
  if (want_qk && !has_qk)
    DLO_FAIL(DLO_ERR_INVALID, "forward: DLO_FWD_QK_NORM without both q/k norm gains in the plan");
  if (!want_qk && (plan->role[R_QNORM] >= 0 || plan->role[R_KNORM] >= 0))
    DLO_FAIL(DLO_ERR_INVALID, "forward: the plan has q/k norm gains but the configuration "
                              "lacks DLO_FWD_QK_NORM");
  return DLO_OK;
}

// Launch overlap by block size: measured on GB300 (forward alone, three
// interleaved rounds), it shortens a small, launch-bound block (hidden 1024,
// 1024 tokens: 80.4 -> 78.6 us) and slows the largest (hidden 6144, 8192
// tokens: 5.57 -> 5.65 ms; hidden 3840, 4096 tokens: unchanged), so by
// default it is on only below 1e11 FLOPs per block.
bool overlap_for(const dlo_dit_cfg& c) {
  const int mode = launch_overlap_mode();
  if (mode >= 0) return mode == 1;
  const double T = static_cast<double>(c.batch) * c.tokens, d = c.hidden, f = c.mlp;
  const double flops = 2.0 * T * (4.0 * d * d + 2.0 * d * f) +
                       4.0 * static_cast<double>(c.batch) * c.tokens * c.tokens * d;
  return flops < 1e11;
}

dlo_status launch_all(const dlo_dit_cfg* cfg, const dlo_plan* plan, const ScratchLayout& sl,
                      const void* block_base, float* x, void* scratch, cudaStream_t stream) {
  const uint8_t* base = static_cast<const uint8_t*>(block_base);
  auto W = [&](int role) { return base + plan->params[plan->role[role]].slot_offset; };
  auto F = [&](int role) { return reinterpret_cast<const float*>(W(role)); };
  auto H = [&](int role) { return reinterpret_cast<const uint16_t*>(W(role)); };
  // optional parameters: null when absent
  auto HO = [&](int role) { return plan->role[role] >= 0 ? H(role) : nullptr; };
  uint8_t* s = static_cast<uint8_t*>(scratch);
  uint16_t* h = reinterpret_cast<uint16_t*>(s + sl.h);
  uint16_t* qkv = reinterpret_cast<uint16_t*>(s + sl.qkv);
  uint16_t* vt = reinterpret_cast<uint16_t*>(s + sl.vt);
  uint16_t* o = reinterpret_cast<uint16_t*>(s + sl.o);
  uint16_t* u = reinterpret_cast<uint16_t*>(s + sl.u);
  float* ws = sl.ws_bytes ? reinterpret_cast<float*>(s + sl.ws) : nullptr;
  const int64_t M = static_cast<int64_t>(cfg->batch) * cfg->tokens;
  const int64_t d = cfg->hidden, f = cfg->mlp;
  // the first kernel follows whatever the stream ran before; each later one
  // follows the previous kernel of this block and may overlap its drain
  DLO_TRY(launch_rmsnorm_mod(x, M, d, F(R_G1), F(R_SHIFT1), F(R_SCALE1), cfg->eps, h, stream));
  PdlScope overlap(overlap_for(*cfg));
  EpiArgs qa{};
  qa.out = qkv;
  qa.vt = vt;
  qa.vt_ld = sl.vt_ld;
  qa.tokens = cfg->tokens;
  qa.v_col0 = static_cast<int>(2 * d);
  qa.ws = ws;
  qa.ws_bytes = sl.ws_bytes;
  qa.bias = HO(R_BQKV);
  DLO_TRY(launch_linear_ex(h, M, d, H(R_WQKV), 3 * d, EPI_QKV, qa, stream));
  if (cfg->flags & (DLO_FWD_QK_NORM | DLO_FWD_ROPE))
    DLO_TRY(launch_qk_norm_rope(qkv, cfg->batch, cfg->tokens, d, cfg->heads,
                                (cfg->flags & DLO_FWD_QK_NORM) ? F(R_QNORM) : nullptr,
                                (cfg->flags & DLO_FWD_QK_NORM) ? F(R_KNORM) : nullptr, cfg->eps,
                                (cfg->flags & DLO_FWD_ROPE) ? kRopeBase : 0.f, stream));
  DLO_TRY(launch_attention_vt(qkv, vt, sl.vt_ld, cfg->batch, cfg->tokens, d, cfg->heads, o, ws,
                              sl.ws_bytes, stream));
  DLO_TRY(launch_linear(o, M, d, H(R_WO), d, EPI_RESID_F32, x, F(R_GATE1), HO(R_BO), ws,
                        sl.ws_bytes, stream));
  DLO_TRY(launch_rmsnorm_mod(x, M, d, F(R_G2), F(R_SHIFT2), F(R_SCALE2), cfg->eps, h, stream));
  DLO_TRY(launch_linear(h, M, d, H(R_W1), f, EPI_GELU_BF16, u, nullptr, HO(R_B1), ws,
                        sl.ws_bytes, stream));
  DLO_TRY(launch_linear(u, M, f, H(R_W2), d, EPI_RESID_F32, x, F(R_GATE2), HO(R_B2), ws,
                        sl.ws_bytes, stream));
  return DLO_OK;
}

// Cached CUDA graphs of the block's launches.  A graph bakes in every kernel
// argument (tensor maps included), so its key is everything those depend
// on: the shape, the plan (by id: addresses of freed plans can be reused),
// the weight base, x, scratch, the device and the GEMM kernel choice.
struct GraphKey {
  int32_t batch, tokens, hidden, heads, mlp, flags;
  float eps;
  uint64_t plan_id;
  const void* base;
  const float* x;
  const void* scratch;
  int device;
  int gemm_mode;
  int overlap;
  bool operator==(const GraphKey& o) const {
    return batch == o.batch && tokens == o.tokens && hidden == o.hidden && heads == o.heads &&
           mlp == o.mlp && flags == o.flags && eps == o.eps && plan_id == o.plan_id && base == o.base &&
           x == o.x && scratch == o.scratch && device == o.device && gemm_mode == o.gemm_mode &&
           overlap == o.overlap;
  }
};

constexpr size_t kMaxGraphs = 1024;
std::mutex g_graph_mu;
std::vector<std::pair<GraphKey, cudaGraphExec_t>> g_graphs;
cudaStream_t g_capture[64] = {};

dlo_status forward_graph(const dlo_dit_cfg* cfg, const dlo_plan* plan, const ScratchLayout& sl,
                         const void* block_base, float* x, void* scratch,
                         cudaStream_t stream) {
  int dev = 0;
  DLO_CUDA(cudaGetDevice(&dev));
  if (dev < 0 || dev >= 64) DLO_FAIL(DLO_ERR_INVALID, "forward: device %d out of range", dev);
  const GraphKey key{cfg->batch, cfg->tokens, cfg->hidden, cfg->heads, cfg->mlp,
                     cfg->flags & ~static_cast<int32_t>(DLO_FWD_GRAPH), cfg->eps, plan->id,
                     block_base, x, scratch, dev, gemm_pair_mode(), overlap_for(*cfg) ? 1 : 0};
  cudaGraphExec_t exec = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_graph_mu);
    for (auto& kv : g_graphs)
      if (kv.first == key) {
        exec = kv.second;
        break;
      }
    if (!exec) {
      if (!g_capture[dev]) DLO_CUDA(cudaStreamCreateWithFlags(&g_capture[dev],
                                                              cudaStreamNonBlocking));
      cudaStream_t cap = g_capture[dev];
      DLO_CUDA(cudaStreamBeginCapture(cap, cudaStreamCaptureModeThreadLocal));
      const dlo_status st = launch_all(cfg, plan, sl, block_base, x, scratch, cap);
      cudaGraph_t graph = nullptr;
      const cudaError_t ce = cudaStreamEndCapture(cap, &graph);
      if (st != DLO_OK) {
        if (graph) cudaGraphDestroy(graph);
        return st;
      }
      DLO_CUDA(ce);
      const cudaError_t ie = cudaGraphInstantiate(&exec, graph, 0);
      cudaGraphDestroy(graph);
      DLO_CUDA(ie);
      if (g_graphs.size() >= kMaxGraphs) {
        // evict the oldest half; wait for the device so none is in flight
        DLO_CUDA(cudaDeviceSynchronize());
        for (size_t i = 0; i < kMaxGraphs / 2; ++i) cudaGraphExecDestroy(g_graphs[i].second);
        g_graphs.erase(g_graphs.begin(), g_graphs.begin() + kMaxGraphs / 2);
      }
      g_graphs.emplace_back(key, exec);
    }
  }
  DLO_CUDA(cudaGraphLaunch(exec, stream));
  return DLO_OK;
}

}  // namespace

dlo_status preload_kernels() {
  static std::once_flag once;
  static dlo_status st = DLO_OK;
  std::call_once(once, [] {
    st = gemm_preload();
    if (st == DLO_OK) st = attention_preload();
    if (st == DLO_OK) st = copy_preload();
    if (st == DLO_OK && !device_error_word()) {
      set_error("cannot resolve the device error word");
      st = DLO_ERR_CUDA;
    }
  });
  return st;
}

dlo_status forward_impl(const dlo_dit_cfg* cfg, const dlo_plan* plan, const void* block_base,
                        float* x, void* scratch, size_t scratch_bytes, cudaStream_t stream) {
  DLO_TRY(check_cfg(cfg));
  TraceRange range("forward", static_cast<int64_t>(cfg->batch) * cfg->tokens);
  DLO_TRY(check_plan(*cfg, plan));
  const ScratchLayout sl = scratch_layout(*cfg);
  if (!block_base || !x || !scratch) DLO_FAIL(DLO_ERR_INVALID, "forward: null pointer");
  if (reinterpret_cast<uintptr_t>(block_base) & 255u)
    DLO_FAIL(DLO_ERR_INVALID, "forward: block base must be 256-byte aligned");
  if ((reinterpret_cast<uintptr_t>(x) & 15u) || (reinterpret_cast<uintptr_t>(scratch) & 255u))
    DLO_FAIL(DLO_ERR_INVALID, "forward: x must be 16-byte and scratch 256-byte aligned");
  if (scratch_bytes < sl.total)
    DLO_FAIL(DLO_ERR_NOMEM, "forward: scratch holds %zu bytes, needs %zu", scratch_bytes,
             sl.total);
  DLO_TRY(preload_kernels());
  if (cfg->flags & DLO_FWD_GRAPH)
    return forward_graph(cfg, plan, sl, block_base, x, scratch, stream);
  return launch_all(cfg, plan, sl, block_base, x, scratch, stream);
}

}  // namespace dlo

extern "C" {

size_t dlo_forward_scratch_bytes(const dlo_dit_cfg* cfg) {
  if (dlo::check_cfg(cfg) != DLO_OK) return 0;
  return dlo::scratch_layout(*cfg).total;
}

int32_t dlo_forward_launches(const dlo_dit_cfg* cfg) {
  using namespace dlo;
  if (check_cfg(cfg) != DLO_OK) return 0;
  const int64_t M = static_cast<int64_t>(cfg->batch) * cfg->tokens, d = cfg->hidden,
                f = cfg->mlp;
  // norm x2, attention (+ the merge of its KV slices), the four linears (+ a
  // reduction each when split), as launch_all issues them
  int32_t n = 2 + attention_plan(cfg->batch, cfg->tokens, d, cfg->heads).launches;
  if (cfg->flags & (DLO_FWD_QK_NORM | DLO_FWD_ROPE)) ++n;   // q/k norm and rotary embedding
  n += linear_plan(M, 3 * d, d, EPI_QKV).launches;
  n += linear_plan(M, d, d, EPI_RESID_F32).launches;
  n += linear_plan(M, f, d, EPI_GELU_BF16).launches;
  n += linear_plan(M, d, f, EPI_RESID_F32).launches;
  return n;
}

dlo_status dlo_forward(const dlo_dit_cfg* cfg, const dlo_plan* plan, const void* block_base,
                       float* x, void* scratch, size_t scratch_bytes, void* stream) {
  return dlo::forward_impl(cfg, plan, block_base, x, scratch, scratch_bytes,
                           static_cast<cudaStream_t>(stream));
}

dlo_status dlo_op_rmsnorm_mod(const float* x, int64_t rows, int64_t d, const float* g,
                              const float* shift, const float* scale, float eps, uint16_t* h,
                              void* stream) {
  return dlo::launch_rmsnorm_mod(x, rows, d, g, shift, scale, eps, h,
                                 static_cast<cudaStream_t>(stream));
}

size_t dlo_op_linear_workspace_bytes(int64_t M, int64_t N, int64_t K, int32_t epilogue) {
  if (M <= 0 || N <= 0 || K <= 0) return 0;
  return dlo::linear_workspace_bytes(M, N, K, epilogue);
}

dlo_status dlo_op_linear(const uint16_t* a, int64_t M, int64_t K, const uint16_t* w, int64_t N,
                         int32_t epilogue, void* out, const float* gate, const uint16_t* bias,
                         void* workspace, size_t workspace_bytes, void* stream) {
  DLO_TRY(dlo::preload_kernels());
  return dlo::launch_linear(a, M, K, w, N, epilogue, out, gate, bias,
                            static_cast<float*>(workspace), workspace_bytes,
                            static_cast<cudaStream_t>(stream));
}

dlo_status dlo_set_gemm_pair_mode(int32_t mode) { return dlo::set_gemm_pair_mode(mode); }

int32_t dlo_op_linear_on_pairs(int64_t M, int64_t N, int64_t K, int32_t epilogue) {
  if (M <= 0 || N <= 0 || K <= 0) return 0;
  return dlo::linear_plan(M, N, K, epilogue).pair;
}

dlo_status dlo_op_qk_norm_rope(uint16_t* qkv, int64_t batch, int64_t tokens, int64_t d,
                               int64_t heads, const float* gq, const float* gk, float eps,
                               float rope_base, void* stream) {
  return dlo::launch_qk_norm_rope(qkv, batch, tokens, d, heads, gq, gk, eps, rope_base,
                                  static_cast<cudaStream_t>(stream));
}

size_t dlo_op_attention_scratch_bytes(int64_t batch, int64_t tokens, int64_t d) {
  if (batch <= 0 || tokens <= 0 || d <= 0) return 0;
  // V transposed, then the KV-slice workspace of either head dim
  const size_t vt = static_cast<size_t>(batch * d * dlo::vt_ld_for(tokens) * 2);
  size_t ws = 0;
  for (int64_t hd : {64, 128})
    if (d % hd == 0) ws = std::max(ws, dlo::attention_plan(batch, tokens, d, d / hd).ws_bytes);
  return (vt + 255) / 256 * 256 + ws;
}

dlo_status dlo_op_attention(const uint16_t* qkv, int64_t batch, int64_t tokens, int64_t d,
                            int64_t heads, uint16_t* o, void* scratch, size_t scratch_bytes,
                            void* stream) {
  using namespace dlo;
  if (batch == 0 || tokens == 0) return DLO_OK;
  const size_t need = dlo_op_attention_scratch_bytes(batch, tokens, d);
  if (!scratch || (reinterpret_cast<uintptr_t>(scratch) & 15u))
    DLO_FAIL(DLO_ERR_INVALID, "dlo_op_attention: scratch must be 16-byte aligned");
  if (scratch_bytes < need)
    DLO_FAIL(DLO_ERR_NOMEM, "dlo_op_attention: scratch holds %zu bytes, needs %zu",
             scratch_bytes, need);
  DLO_TRY(preload_kernels());
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint16_t* vt = static_cast<uint16_t*>(scratch);
  const int64_t vt_ld = vt_ld_for(tokens);
  const size_t vt_bytes = (static_cast<size_t>(batch * d * vt_ld * 2) + 255) / 256 * 256;
  float* ws = reinterpret_cast<float*>(static_cast<uint8_t*>(scratch) + vt_bytes);
  DLO_TRY(launch_transpose_v(qkv, batch, tokens, d, vt, vt_ld, st));
  return launch_attention_vt(qkv, vt, vt_ld, batch, tokens, d, heads, o, ws,
                             scratch_bytes - vt_bytes, st);
}

}  // extern "C"
