// dlo_oracle.cpp — TEST INFRASTRUCTURE ONLY.
//
// A plain, slow, obviously-correct CPU statement of what the double-buffered
// per-block weight stream of Distributed Layerwise Offload (DLO) computes.
// It exists so the CUDA path can be checked against something written
// independently of it.  Only the test suite, the smoke check and the CPU
// baseline leg of the benchmark may load this library; the product path
// never does, and this file shares no code, header or table with the CUDA
// library.
//
// Sources (cited by page title and section):
//   [B1] "Distributed Layerwise Offload" (vLLM blog preview, 2026-07-30):
//        "Weight Sharding + AllGather", "Double-Buffer Memory Bound",
//        "Slot Tracking: i%2 + Dynamic Correction".
//   [B2] "Distributed Layerwise Offload: Scaling Toward 200B+ DiT Models
//        Efficiently in vLLM-Omni" (vLLM blog, 2026-08-17):
//        "2. Weight Sharding with AllGather Reconstruction",
//        "3. Double-Buffered Prefetch with H2D + AllGather Overlap".
//   [D5] vLLM-Omni design doc "Distributed Layerwise Offload": "AllGather path".
//
// The pages never define the transformer block that consumes the streamed
// weights.  The block below is the synthetic DiT block the workload
// specifies (RMSNorm, adaLN shift/scale/gate, QKV linear, softmax attention,
// out-projection, GELU-tanh MLP); its readings are listed with each function.
// The checkpoint-shaped variant adds what real DiT checkpoints carry and the
// pages do not define either: biases on the four linears, a per-head RMSNorm
// of q and k with learned gains, and rotary position embedding of q and k
// (plainest readings, stated with oracle_qk_norm and oracle_rope).
//
// Arithmetic: every floating-point step runs in IEEE double.  Weights arrive
// as float (bf16 values widened exactly).  Threads split independent output
// rows only; no reduction is reordered.
//
// Parity status: sharding, reassembly, slot layout and the schedule are
// pinned by tests against the pages' closed forms and invariants; the block
// forward is pinned by closed-form special cases (zero gates, uniform
// attention, permutation weights, one token) and by library routines on
// small shapes.

#include <cmath>
#include <cstdint>
#include <cstring>
#include <thread>
#include <vector>
#include <algorithm>
#include <functional>

extern "C" {

// ---------------------------------------------------------------------------
// Sharding: [B2] §2 shows the shard length as a ceiling division of the flat
// element count by the data-parallel size, with zero padding so that every
// shard has the same length (a requirement of all_gather_into_tensor), and
// rank r holding the flat window [r*S, (r+1)*S).
// ---------------------------------------------------------------------------

// Storage extent, in elements, of a view with the given extents and element
// strides.  [D5] "Request and loading constraints": finalized 1-byte weights
// and their scales may be contiguous or transposed views, and they are
// packed in physical order.  Reading: the packed elements of a view are its
// storage from element [0,..,0] through its last element in memory, i.e.
// 1 + sum_i (shape_i - 1) * stride_i (strides >= 0); for row-major strides
// that is the element count.
int64_t oracle_storage_extent(int32_t ndim, const int64_t* shape, const int64_t* stride) {
  int64_t last = 0;
  for (int32_t i = 0; i < ndim; ++i) last += (shape[i] - 1) * stride[i];
  return last + 1;
}

int64_t oracle_shard_numel(int64_t total_numel, int32_t dp_size) {
  if (dp_size <= 0 || total_numel < 0) return -1;
  return (total_numel + dp_size - 1) / dp_size;
}

// Flatten: [B1] "Weight Sharding + AllGather" — a block's parameters are
// flattened by dtype.  Reading: parameters of one dtype are concatenated in
// registration order with no gap.  Copies the parameters whose dtype code
// equals `dtype` into `out` and returns the number of elements written.
int64_t oracle_flatten_group(const void* const* params, const int64_t* numels,
                             const int32_t* dtypes, int32_t n_params,
                             int32_t dtype, int32_t esize, void* out) {
  int64_t at = 0;
  for (int32_t p = 0; p < n_params; ++p) {
    if (dtypes[p] != dtype) continue;
    std::memcpy(static_cast<uint8_t*>(out) + at * esize, params[p],
                static_cast<size_t>(numels[p]) * esize);
    at += numels[p];
  }
  return at;
}

// Shard r receives flat[r*S, min((r+1)*S, N)); the rest of its S elements
// stay zero ([B2] §2: a zero tensor of shard length, then a copy of the
// window that lies inside the flat view).
void oracle_shard(const void* flat, int64_t numel, int32_t esize,
                  int32_t dp_size, void* const* shards_out) {
  const int64_t S = oracle_shard_numel(numel, dp_size);
  for (int32_t r = 0; r < dp_size; ++r) {
    uint8_t* dst = static_cast<uint8_t*>(shards_out[r]);
    std::memset(dst, 0, static_cast<size_t>(S) * esize);
    const int64_t lo = static_cast<int64_t>(r) * S;
    const int64_t hi = std::min(lo + S, numel);
    for (int64_t e = lo; e < hi; ++e)
      std::memcpy(dst + (e - lo) * esize,
                  static_cast<const uint8_t*>(flat) + e * esize, esize);
  }
}

// Reassembly, [B1] "Weight Sharding + AllGather" step 2 and [D5] "AllGather
// path": all_gather_into_tensor concatenates the equal shards in rank
// order.  Output holds dp_size*S elements, padding included.
void oracle_reassemble(const void* const* shards, int64_t shard_numel,
                       int32_t esize, int32_t dp_size, void* gathered_out) {
  for (int32_t r = 0; r < dp_size; ++r)
    for (int64_t e = 0; e < shard_numel; ++e)
      std::memcpy(static_cast<uint8_t*>(gathered_out) +
                      (static_cast<int64_t>(r) * shard_numel + e) * esize,
                  static_cast<const uint8_t*>(shards[r]) + e * esize, esize);
}

// Slot image: where each dtype group's gathered buffer lives inside one
// device slot.  [B2] §3 sizes a slot to the largest block; the pages do not
// say how several dtype groups share it.  Reading: groups are placed in the
// order in which their dtype first appears in registration order, each
// starting at a multiple of `align` bytes, each occupying dp_size*S_g
// elements.  Writes group_base[g] for the first n_groups groups and returns
// the slot's used byte count (end of the last group).
int64_t oracle_slot_layout(const int64_t* numels, const int32_t* dtypes,
                           const int32_t* esizes, int32_t n_params,
                           int32_t dp_size, int64_t align,
                           int32_t* group_dtype_out, int64_t* group_base_out,
                           int32_t* n_groups_out) {
  std::vector<int32_t> order;
  for (int32_t p = 0; p < n_params; ++p)
    if (std::find(order.begin(), order.end(), dtypes[p]) == order.end())
      order.push_back(dtypes[p]);
  int64_t cursor = 0;
  for (size_t g = 0; g < order.size(); ++g) {
    int64_t n = 0;
    int32_t es = 0;
    for (int32_t p = 0; p < n_params; ++p)
      if (dtypes[p] == order[g]) { n += numels[p]; es = esizes[p]; }
    int64_t base = (cursor + align - 1) / align * align;
    group_dtype_out[g] = order[g];
    group_base_out[g] = base;
    cursor = base + dp_size * oracle_shard_numel(n, dp_size) * es;
  }
  *n_groups_out = static_cast<int32_t>(order.size());
  return cursor;
}

// ---------------------------------------------------------------------------
// Slot schedule: [B1] "Slot Tracking: i%2 + Dynamic Correction" and
// "Weight Sharding + AllGather"; [B2] §3.  Simulated literally: one hook per
// block, chained circularly (hook 0's predecessor is hook n-1, so that the
// tail->head wrap is corrected), current_slot initialised to i % 2,
// _prefetched_slot unset.  Before each forward the hook adopts its
// predecessor's _prefetched_slot when that is set, waits for the slot's
// ready event, prefetches block (i+1) mod n into the other slot (after the
// free event of the forward that last read that slot — a write-after-read
// wait the pages do not draw but which the reuse of two buffers requires),
// records _prefetched_slot, runs, and records the free event of its slot.
// A setup prefetch places block 0 in slot 0 before the first forward.
//
// Output per forward k (7 int32 each):
//   k, block, read_slot, prefetch_block, prefetch_slot,
//   waits_on_free_of_k (-1 if the slot was never read), violation flags
// violation flags: bit0 = read slot does not hold the block,
//                  bit1 = prefetch targets the slot being read,
//                  bit2 = more than two blocks resident (cannot happen with
//                         two slots; kept as an explicit check).
// `use_correction` = 0 disables the _prefetched_slot adoption (used by
// tests to show the collision the correction exists to prevent).
// Returns the number of forwards written.
int32_t oracle_schedule(int32_t n_blocks, int32_t n_steps,
                        int32_t use_correction, int32_t* out) {
  if (n_blocks <= 0 || n_steps < 0) return -1;
  struct Hook { int32_t index, current_slot, prefetched_slot, prev; };
  std::vector<Hook> hooks(n_blocks);
  for (int32_t i = 0; i < n_blocks; ++i)
    hooks[i] = {i, i % 2, -1, (i + n_blocks - 1) % n_blocks};
  int32_t slot_holds[2] = {0, -1};     // setup prefetch: block 0 -> slot 0
  int32_t last_reader[2] = {-1, -1};   // forward index that last read a slot
  int32_t k = 0;
  for (int32_t step = 0; step < n_steps; ++step) {
    for (int32_t i = 0; i < n_blocks; ++i, ++k) {
      Hook& h = hooks[i];
      const Hook& prev = hooks[h.prev];
      if (use_correction && prev.prefetched_slot >= 0)
        h.current_slot = prev.prefetched_slot;
      int32_t flags = 0;
      if (slot_holds[h.current_slot] != i) flags |= 1;
      const int32_t next_block = (i + 1) % n_blocks;
      const int32_t next_slot = 1 - h.current_slot;
      if (next_slot == h.current_slot) flags |= 2;
      const int32_t waits_on = last_reader[next_slot];
      slot_holds[next_slot] = next_block;
      h.prefetched_slot = next_slot;
      last_reader[h.current_slot] = k;
      int32_t* e = out + 7 * k;
      e[0] = k; e[1] = i; e[2] = h.current_slot; e[3] = next_block;
      e[4] = next_slot; e[5] = waits_on; e[6] = flags;
    }
  }
  return k;
}

// ---------------------------------------------------------------------------
// Synthetic DiT block (not on the pages).  Readings:
//   RMSNorm(x) = x / sqrt(mean(x^2) + eps), times gain g;
//   adaLN modulation  h = RMSNorm(x)*g*(1+scale) + shift;
//   linear weights in [out, in] layout, no biases: y[t,n] = sum_k a[t,k] W[n,k];
//   qkv = h Wqkv^T, columns [0,d) = Q, [d,2d) = K, [2d,3d) = V, head j owning
//   columns [j*hd, (j+1)*hd) of each; non-causal softmax attention per head
//   with scale 1/sqrt(hd); no positional encoding, no QK-norm;
//   x += gate1 * (o Wo^T);  h2 = RMSNorm(x)*g2*(1+scale2)+shift2;
//   x += gate2 * (GELU_tanh(h2 W1^T) W2^T);
//   GELU_tanh(z) = 0.5 z (1 + tanh(sqrt(2/pi) (z + 0.044715 z^3))).
// ---------------------------------------------------------------------------

}  // extern "C"

// Splits [0, rows) into contiguous ranges, one per thread.
static void run_rows(int64_t rows, int32_t threads,
                     const std::function<void(int64_t, int64_t)>& body) {
  if (threads <= 1 || rows < 2) { body(0, rows); return; }
  const int32_t nt = static_cast<int32_t>(std::min<int64_t>(threads, rows));
  std::vector<std::thread> pool;
  const int64_t per = (rows + nt - 1) / nt;
  for (int32_t t = 0; t < nt; ++t) {
    const int64_t lo = t * per, hi = std::min(rows, lo + per);
    if (lo >= hi) break;
    pool.emplace_back([&body, lo, hi] { body(lo, hi); });
  }
  for (auto& th : pool) th.join();
}

// One head's hd values v <- v / sqrt(mean(v^2) + eps) * g (the per-head
// q/k RMSNorm of the checkpoint-shaped block).
static void qk_norm_head(double* v, int64_t hd, const float* g, double eps) {
  double ss = 0.0;
  for (int64_t c = 0; c < hd; ++c) ss += v[c] * v[c];
  const double inv = 1.0 / std::sqrt(ss / static_cast<double>(hd) + eps);
  for (int64_t c = 0; c < hd; ++c) v[c] = v[c] * inv * static_cast<double>(g[c]);
}

// One head's values at position pos rotated pair by pair: pair (2i, 2i+1)
// by the angle pos * base^(-2i/hd) (RoFormer's rotary embedding).
static void rope_head(double* v, int64_t hd, double pos, double base) {
  for (int64_t i = 0; i < hd / 2; ++i) {
    const double ang = pos * std::pow(base, -2.0 * static_cast<double>(i) /
                                                static_cast<double>(hd));
    const double c = std::cos(ang), s = std::sin(ang);
    const double a0 = v[2 * i], b0 = v[2 * i + 1];
    v[2 * i] = a0 * c - b0 * s;
    v[2 * i + 1] = a0 * s + b0 * c;
  }
}

extern "C" {

double oracle_gelu_tanh(double z) {
  const double c = std::sqrt(2.0 / std::acos(-1.0));
  return 0.5 * z * (1.0 + std::tanh(c * (z + 0.044715 * z * z * z)));
}

// out[e] = oracle_gelu_tanh(z[e]) for e < n (the block's MLP activation,
// element by element).
void oracle_gelu_tanh_array(const double* z, int64_t n, double* out) {
  for (int64_t e = 0; e < n; ++e) out[e] = oracle_gelu_tanh(z[e]);
}

// h[t,:] = x[t,:] / sqrt(mean(x[t,:]^2) + eps) * g * (1 + scale) + shift
void oracle_rmsnorm_mod(const double* x, int64_t rows, int64_t d,
                        const float* g, const float* shift, const float* scale,
                        double eps, double* h_out) {
  for (int64_t t = 0; t < rows; ++t) {
    const double* xr = x + t * d;
    double ss = 0.0;
    for (int64_t c = 0; c < d; ++c) ss += xr[c] * xr[c];
    const double inv = 1.0 / std::sqrt(ss / static_cast<double>(d) + eps);
    for (int64_t c = 0; c < d; ++c)
      h_out[t * d + c] = xr[c] * inv * static_cast<double>(g[c]) *
                             (1.0 + static_cast<double>(scale[c])) +
                         static_cast<double>(shift[c]);
  }
}

// y[t,n] = sum_k a[t,k] * w[n,k]   (w in [out, in] layout)
void oracle_linear(const double* a, int64_t rows, int64_t k_dim,
                   const float* w, int64_t n_dim, double* y, int32_t threads) {
  run_rows(rows, threads, [&](int64_t lo, int64_t hi) {
    for (int64_t t = lo; t < hi; ++t) {
      const double* ar = a + t * k_dim;
      for (int64_t n = 0; n < n_dim; ++n) {
        const float* wr = w + n * k_dim;
        double acc = 0.0;
        for (int64_t k = 0; k < k_dim; ++k)
          acc += ar[k] * static_cast<double>(wr[k]);
        y[t * n_dim + n] = acc;
      }
    }
  });
}

// Softmax attention, non-causal, per batch item and head.
// qkv: [batch*tokens, 3d]; o: [batch*tokens, d].
void oracle_attention(const double* qkv, int64_t batch, int64_t tokens,
                      int64_t d, int64_t heads, double* o, int32_t threads) {
  const int64_t hd = d / heads;
  const double scale = 1.0 / std::sqrt(static_cast<double>(hd));
  const int64_t ld = 3 * d;
  run_rows(batch * heads * tokens, threads, [&](int64_t lo, int64_t hi) {
    std::vector<double> s(tokens);
    for (int64_t job = lo; job < hi; ++job) {
      const int64_t b = job / (heads * tokens);
      const int64_t j = (job / tokens) % heads;
      const int64_t t = job % tokens;
      const double* q = qkv + (b * tokens + t) * ld + j * hd;
      double m = -INFINITY;
      for (int64_t u = 0; u < tokens; ++u) {
        const double* kk = qkv + (b * tokens + u) * ld + d + j * hd;
        double dot = 0.0;
        for (int64_t c = 0; c < hd; ++c) dot += q[c] * kk[c];
        s[u] = dot * scale;
        m = std::max(m, s[u]);
      }
      double denom = 0.0;
      for (int64_t u = 0; u < tokens; ++u) { s[u] = std::exp(s[u] - m); denom += s[u]; }
      double* orow = o + (b * tokens + t) * d + j * hd;
      for (int64_t c = 0; c < hd; ++c) {
        double acc = 0.0;
        for (int64_t u = 0; u < tokens; ++u)
          acc += s[u] * qkv[(b * tokens + u) * ld + 2 * d + j * hd + c];
        orow[c] = acc / denom;
      }
    }
  });
}

// Per-head RMSNorm of q and k (the checkpoint-shaped block): for every row
// and head j, q_j <- q_j / sqrt(mean(q_j^2) + eps) * gq and likewise k_j
// with gk, each over the head's hd values; gq, gk: [hd].  qkv: [rows, 3d],
// q in columns [0, d), k in [d, 2d); v untouched.
void oracle_qk_norm(double* qkv, int64_t rows, int64_t d, int64_t heads, const float* gq,
                    const float* gk, double eps) {
  const int64_t hd = d / heads;
  for (int64_t t = 0; t < rows; ++t)
    for (int64_t part = 0; part < 2; ++part)
      for (int64_t j = 0; j < heads; ++j)
        qk_norm_head(qkv + t * 3 * d + part * d + j * hd, hd, part == 0 ? gq : gk, eps);
}

// Rotary position embedding of q and k (the checkpoint-shaped block), in the
// form of Su et al., "RoFormer": the head's values are taken in pairs
// (2i, 2i+1), i = 0 .. hd/2 - 1, and the pair of the token at position p is
// rotated by the angle p * base^(-2i/hd):
//   (a, b) <- (a cos - b sin, a sin + b cos).
// The position is the token's index within its batch item (1-D positions).
void oracle_rope(double* qkv, int64_t batch, int64_t tokens, int64_t d, int64_t heads,
                 double base) {
  const int64_t hd = d / heads;
  for (int64_t r = 0; r < batch * tokens; ++r) {
    const double pos = static_cast<double>(r % tokens);
    for (int64_t part = 0; part < 2; ++part)
      for (int64_t j = 0; j < heads; ++j) rope_head(qkv + r * 3 * d + part * d + j * hd, hd, pos, base);
  }
}

// The block forward with the checkpoint-shaped additions, each optional
// (null / 0 = absent): biases bqkv[3d], bo[d], b1[f], b2[d] added to the
// linears' outputs (before the GELU and before the gates); q/k RMSNorm gains
// gq, gk [hd] (both or neither), applied after the QKV bias; RoPE with
// rope_base > 0, applied after the q/k norm.  Order of operations:
//   h = rmsnorm_mod(x); qkv = h Wqkv^T + bqkv; qk-norm; rope; o = attention
//   x += gate1 * (o Wo^T + bo)
//   h2 = rmsnorm_mod(x); x += gate2 * (gelu(h2 W1^T + b1) W2^T + b2)
void oracle_block_forward_ex(const float* x_in, int64_t batch, int64_t tokens, int64_t d,
                             int64_t heads, int64_t f, double eps, const float* const* p,
                             const float* bqkv, const float* bo, const float* b1,
                             const float* b2, const float* gq, const float* gk,
                             double rope_base, double* x_out, int32_t threads) {
  const int64_t M = batch * tokens;
  std::vector<double> x(M * d), h(M * d), qkv(M * 3 * d), o(M * d), y(M * d), u(M * f);
  for (int64_t e = 0; e < M * d; ++e) x[e] = static_cast<double>(x_in[e]);
  auto add_bias = [](double* v, int64_t rows, int64_t n, const float* b) {
    if (!b) return;
    for (int64_t t = 0; t < rows; ++t)
      for (int64_t c = 0; c < n; ++c) v[t * n + c] += static_cast<double>(b[c]);
  };
  // attention branch
  oracle_rmsnorm_mod(x.data(), M, d, p[0], p[1], p[2], eps, h.data());
  oracle_linear(h.data(), M, d, p[4], 3 * d, qkv.data(), threads);
  add_bias(qkv.data(), M, 3 * d, bqkv);
  if (gq && gk) oracle_qk_norm(qkv.data(), M, d, heads, gq, gk, eps);
  if (rope_base > 0.0) oracle_rope(qkv.data(), batch, tokens, d, heads, rope_base);
  oracle_attention(qkv.data(), batch, tokens, d, heads, o.data(), threads);
  oracle_linear(o.data(), M, d, p[5], d, y.data(), threads);
  add_bias(y.data(), M, d, bo);
  for (int64_t t = 0; t < M; ++t)
    for (int64_t c = 0; c < d; ++c)
      x[t * d + c] += static_cast<double>(p[3][c]) * y[t * d + c];
  // MLP branch
  oracle_rmsnorm_mod(x.data(), M, d, p[6], p[7], p[8], eps, h.data());
  oracle_linear(h.data(), M, d, p[10], f, u.data(), threads);
  add_bias(u.data(), M, f, b1);
  for (int64_t e = 0; e < M * f; ++e) u[e] = oracle_gelu_tanh(u[e]);
  oracle_linear(u.data(), M, f, p[11], d, y.data(), threads);
  add_bias(y.data(), M, d, b2);
  for (int64_t t = 0; t < M; ++t)
    for (int64_t c = 0; c < d; ++c)
      x[t * d + c] += static_cast<double>(p[9][c]) * y[t * d + c];
  std::memcpy(x_out, x.data(), sizeof(double) * M * d);
}

// One block forward.  Parameter order of `p` (all float arrays):
//   0 g1[d]  1 shift1[d]  2 scale1[d]  3 gate1[d]  4 Wqkv[3d,d]  5 Wo[d,d]
//   6 g2[d]  7 shift2[d]  8 scale2[d]  9 gate2[d] 10 W1[f,d]    11 W2[d,f]
// x_in: [batch*tokens, d] float; x_out: same shape, double.
void oracle_block_forward(const float* x_in, int64_t batch, int64_t tokens,
                          int64_t d, int64_t heads, int64_t f, double eps,
                          const float* const* p, double* x_out,
                          int32_t threads) {
  const int64_t M = batch * tokens;
  std::vector<double> x(M * d), h(M * d), qkv(M * 3 * d), o(M * d), y(M * d),
      u(M * f);
  for (int64_t e = 0; e < M * d; ++e) x[e] = static_cast<double>(x_in[e]);
  // attention branch
  oracle_rmsnorm_mod(x.data(), M, d, p[0], p[1], p[2], eps, h.data());
  oracle_linear(h.data(), M, d, p[4], 3 * d, qkv.data(), threads);
  oracle_attention(qkv.data(), batch, tokens, d, heads, o.data(), threads);
  oracle_linear(o.data(), M, d, p[5], d, y.data(), threads);
  for (int64_t t = 0; t < M; ++t)
    for (int64_t c = 0; c < d; ++c)
      x[t * d + c] += static_cast<double>(p[3][c]) * y[t * d + c];
  // MLP branch
  oracle_rmsnorm_mod(x.data(), M, d, p[6], p[7], p[8], eps, h.data());
  oracle_linear(h.data(), M, d, p[10], f, u.data(), threads);
  for (int64_t e = 0; e < M * f; ++e) u[e] = oracle_gelu_tanh(u[e]);
  oracle_linear(u.data(), M, f, p[11], d, y.data(), threads);
  for (int64_t t = 0; t < M; ++t)
    for (int64_t c = 0; c < d; ++c)
      x[t * d + c] += static_cast<double>(p[9][c]) * y[t * d + c];
  std::memcpy(x_out, x.data(), sizeof(double) * M * d);
}


// The same block forward, evaluated only for the query rows listed in
// `rows` (indices into [0, batch*tokens)): every token still contributes
// its K and V to attention, but the out-projection, the residuals and the
// MLP run for the listed rows only.  For a listed row each value is formed
// by exactly the operations, in the same order, as oracle_block_forward.
// Output: x_out[i, :] is the block output of row rows[i].
void oracle_block_forward_rows(const float* x_in, int64_t batch, int64_t tokens, int64_t d,
                               int64_t heads, int64_t f, double eps, const float* const* p,
                               const int64_t* rows, int64_t n_rows, double* x_out,
                               int32_t threads) {
  const int64_t M = batch * tokens;
  const int64_t hd = d / heads;
  const double scale = 1.0 / std::sqrt(static_cast<double>(hd));
  std::vector<double> x(M * d), h(M * d), kv(M * 2 * d);
  for (int64_t e = 0; e < M * d; ++e) x[e] = static_cast<double>(x_in[e]);
  oracle_rmsnorm_mod(x.data(), M, d, p[0], p[1], p[2], eps, h.data());
  // K and V of every token: rows d..3d of Wqkv
  oracle_linear(h.data(), M, d, p[4] + d * d, 2 * d, kv.data(), threads);
  std::vector<double> xs(n_rows * d), hs(n_rows * d), q(n_rows * d), o(n_rows * d),
      y(n_rows * d), u(n_rows * f);
  for (int64_t i = 0; i < n_rows; ++i)
    for (int64_t c = 0; c < d; ++c) {
      xs[i * d + c] = x[rows[i] * d + c];
      hs[i * d + c] = h[rows[i] * d + c];
    }
  oracle_linear(hs.data(), n_rows, d, p[4], d, q.data(), threads);   // Q rows 0..d
  run_rows(n_rows * heads, threads, [&](int64_t lo, int64_t hi) {
    std::vector<double> s(tokens);
    for (int64_t job = lo; job < hi; ++job) {
      const int64_t i = job / heads, j = job % heads;
      const int64_t b = rows[i] / tokens;
      const double* qr = q.data() + i * d + j * hd;
      double m = -INFINITY;
      for (int64_t t = 0; t < tokens; ++t) {
        const double* kk = kv.data() + (b * tokens + t) * 2 * d + j * hd;
        double dot = 0.0;
        for (int64_t c = 0; c < hd; ++c) dot += qr[c] * kk[c];
        s[t] = dot * scale;
        m = std::max(m, s[t]);
      }
      double denom = 0.0;
      for (int64_t t = 0; t < tokens; ++t) { s[t] = std::exp(s[t] - m); denom += s[t]; }
      for (int64_t c = 0; c < hd; ++c) {
        double acc = 0.0;
        for (int64_t t = 0; t < tokens; ++t)
          acc += s[t] * kv[(b * tokens + t) * 2 * d + d + j * hd + c];
        o[i * d + j * hd + c] = acc / denom;
      }
    }
  });
  oracle_linear(o.data(), n_rows, d, p[5], d, y.data(), threads);
  for (int64_t i = 0; i < n_rows; ++i)
    for (int64_t c = 0; c < d; ++c) xs[i * d + c] += static_cast<double>(p[3][c]) * y[i * d + c];
  oracle_rmsnorm_mod(xs.data(), n_rows, d, p[6], p[7], p[8], eps, hs.data());
  oracle_linear(hs.data(), n_rows, d, p[10], f, u.data(), threads);
  for (int64_t e = 0; e < n_rows * f; ++e) u[e] = oracle_gelu_tanh(u[e]);
  oracle_linear(u.data(), n_rows, f, p[11], d, y.data(), threads);
  for (int64_t i = 0; i < n_rows; ++i)
    for (int64_t c = 0; c < d; ++c) xs[i * d + c] += static_cast<double>(p[9][c]) * y[i * d + c];
  std::memcpy(x_out, xs.data(), sizeof(double) * n_rows * d);
}

// oracle_block_forward_ex evaluated only for the listed query rows (as
// oracle_block_forward_rows does for the plain block): every token's K and V
// get their bias, k-norm and rotation, the listed rows' Q likewise, and the
// out-projection, residuals and MLP run for the listed rows only.  Each value
// of a listed row is formed by the same operations, in the same order, as in
// oracle_block_forward_ex.
void oracle_block_forward_ex_rows(const float* x_in, int64_t batch, int64_t tokens, int64_t d,
                                  int64_t heads, int64_t f, double eps, const float* const* p,
                                  const float* bqkv, const float* bo, const float* b1,
                                  const float* b2, const float* gq, const float* gk,
                                  double rope_base, const int64_t* rows, int64_t n_rows,
                                  double* x_out, int32_t threads) {
  const int64_t M = batch * tokens;
  const int64_t hd = d / heads;
  const double scale = 1.0 / std::sqrt(static_cast<double>(hd));
  const bool qk_norm = gq && gk;
  std::vector<double> x(M * d), h(M * d), kv(M * 2 * d);
  for (int64_t e = 0; e < M * d; ++e) x[e] = static_cast<double>(x_in[e]);
  oracle_rmsnorm_mod(x.data(), M, d, p[0], p[1], p[2], eps, h.data());
  // K and V of every token: rows d..3d of Wqkv, their bias, then k's norm
  // and rotation
  oracle_linear(h.data(), M, d, p[4] + d * d, 2 * d, kv.data(), threads);
  for (int64_t t = 0; t < M; ++t) {
    double* r = kv.data() + t * 2 * d;
    if (bqkv)
      for (int64_t c = 0; c < 2 * d; ++c) r[c] += static_cast<double>(bqkv[d + c]);
    for (int64_t j = 0; j < heads; ++j) {
      if (qk_norm) qk_norm_head(r + j * hd, hd, gk, eps);
      if (rope_base > 0.0)
        rope_head(r + j * hd, hd, static_cast<double>(t % tokens), rope_base);
    }
  }
  std::vector<double> xs(n_rows * d), hs(n_rows * d), q(n_rows * d), o(n_rows * d),
      y(n_rows * d), u(n_rows * f);
  for (int64_t i = 0; i < n_rows; ++i)
    for (int64_t c = 0; c < d; ++c) {
      xs[i * d + c] = x[rows[i] * d + c];
      hs[i * d + c] = h[rows[i] * d + c];
    }
  oracle_linear(hs.data(), n_rows, d, p[4], d, q.data(), threads);   // Q rows 0..d
  for (int64_t i = 0; i < n_rows; ++i) {
    double* r = q.data() + i * d;
    if (bqkv)
      for (int64_t c = 0; c < d; ++c) r[c] += static_cast<double>(bqkv[c]);
    for (int64_t j = 0; j < heads; ++j) {
      if (qk_norm) qk_norm_head(r + j * hd, hd, gq, eps);
      if (rope_base > 0.0)
        rope_head(r + j * hd, hd, static_cast<double>(rows[i] % tokens), rope_base);
    }
  }
  run_rows(n_rows * heads, threads, [&](int64_t lo, int64_t hi) {
    std::vector<double> s(tokens);
    for (int64_t job = lo; job < hi; ++job) {
      const int64_t i = job / heads, j = job % heads;
      const int64_t b = rows[i] / tokens;
      const double* qr = q.data() + i * d + j * hd;
      double m = -INFINITY;
      for (int64_t t = 0; t < tokens; ++t) {
        const double* kk = kv.data() + (b * tokens + t) * 2 * d + j * hd;
        double dot = 0.0;
        for (int64_t c = 0; c < hd; ++c) dot += qr[c] * kk[c];
        s[t] = dot * scale;
        m = std::max(m, s[t]);
      }
      double denom = 0.0;
      for (int64_t t = 0; t < tokens; ++t) { s[t] = std::exp(s[t] - m); denom += s[t]; }
      for (int64_t c = 0; c < hd; ++c) {
        double acc = 0.0;
        for (int64_t t = 0; t < tokens; ++t)
          acc += s[t] * kv[(b * tokens + t) * 2 * d + d + j * hd + c];
        o[i * d + j * hd + c] = acc / denom;
      }
    }
  });
  auto add_bias = [](double* v, int64_t n_r, int64_t n, const float* bias) {
    if (!bias) return;
    for (int64_t t = 0; t < n_r; ++t)
      for (int64_t c = 0; c < n; ++c) v[t * n + c] += static_cast<double>(bias[c]);
  };
  oracle_linear(o.data(), n_rows, d, p[5], d, y.data(), threads);
  add_bias(y.data(), n_rows, d, bo);
  for (int64_t i = 0; i < n_rows; ++i)
    for (int64_t c = 0; c < d; ++c) xs[i * d + c] += static_cast<double>(p[3][c]) * y[i * d + c];
  oracle_rmsnorm_mod(xs.data(), n_rows, d, p[6], p[7], p[8], eps, hs.data());
  oracle_linear(hs.data(), n_rows, d, p[10], f, u.data(), threads);
  add_bias(u.data(), n_rows, f, b1);
  for (int64_t e = 0; e < n_rows * f; ++e) u[e] = oracle_gelu_tanh(u[e]);
  oracle_linear(u.data(), n_rows, f, p[11], d, y.data(), threads);
  add_bias(y.data(), n_rows, d, b2);
  for (int64_t i = 0; i < n_rows; ++i)
    for (int64_t c = 0; c < d; ++c) xs[i * d + c] += static_cast<double>(p[9][c]) * y[i * d + c];
  std::memcpy(x_out, xs.data(), sizeof(double) * n_rows * d);
}

}  // extern "C"
