// plan.cpp — the per-block layout and the CPU flatten/pad/split.
//
// "Distributed Layerwise Offload" (vLLM blog preview, 2026-07-30),
// "Weight Sharding + AllGather": a block's parameters are flattened by dtype
// and split into dp_size equal shards kept in pinned host memory.
// "Distributed Layerwise Offload: Scaling Toward 200B+ DiT Models
// Efficiently in vLLM-Omni", "2. Weight Sharding with AllGather
// Reconstruction": shard length = ceil(total / dp_size), zero padding so all
// shards are equal, rank r holds the window [r*S, (r+1)*S).
// Layout readings (the pages are silent): registration order inside a dtype
// group, no gap between parameters; groups in order of first appearance,
// each at a 256-byte aligned base of the slot, each taking n_shards*S_g
// elements (the gathered buffer with its padding).
#include <algorithm>
#include <cstdarg>
#include <cstring>
#include <atomic>
#include <new>

#include "common.h"
#include "trace.h"

namespace dlo {

namespace {
thread_local std::string g_last_error;
}

void set_error(const char* fmt, ...) {
  char buf[1024];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
}

void clear_error() { g_last_error.clear(); }

nvtxDomainHandle_t trace_domain() {
  static const nvtxDomainHandle_t d = nvtxDomainCreateA("dlo");
  return d;
}

const char* const kRoleNames[R_COUNT] = {
    "norm1.weight", "ada1.shift", "ada1.scale", "ada1.gate",
    "attn.qkv.weight", "attn.out.weight",
    "norm2.weight", "ada2.shift", "ada2.scale", "ada2.gate",
    "mlp.fc1.weight", "mlp.fc2.weight",
    "attn.qkv.bias", "attn.out.bias", "mlp.fc1.bias", "mlp.fc2.bias",
    "attn.q_norm.weight", "attn.k_norm.weight"};

static int32_t esize_of(int32_t dtype) {
  switch (dtype) {
    case DLO_BF16: return 2;
    case DLO_F32: return 4;
    case DLO_F16: return 2;
    case DLO_FP8_E4M3:
    case DLO_FP8_E5M2:
    case DLO_I8:
    case DLO_U8:
    case DLO_E8M0: return 1;
    default: return 0;
  }
}

// dtype the block forward reads for each DiT role
static int32_t role_dtype(int r) {
  return (r == R_WQKV || r == R_WO || r == R_W1 || r == R_W2 || r == R_BQKV || r == R_BO ||
          r == R_B1 || r == R_B2)
             ? DLO_BF16
             : DLO_F32;
}

}  // namespace dlo

extern "C" {

const char* dlo_last_error(void) { return dlo::g_last_error.c_str(); }

const char* dlo_version(void) { return "dlo-gb300 0.1 (sm_103a)"; }

dlo_status dlo_plan_create(const dlo_param_desc* params, int32_t n_params,
                           int32_t n_shards, dlo_plan** out) {
  using namespace dlo;
  dlo::TraceRange range("plan_create", n_params);
  if (!params || !out) DLO_FAIL(DLO_ERR_INVALID, "dlo_plan_create: null argument");
  if (n_params < 1) DLO_FAIL(DLO_ERR_INVALID, "dlo_plan_create: n_params must be >= 1");
  if (n_shards < 1) DLO_FAIL(DLO_ERR_INVALID, "dlo_plan_create: n_shards must be >= 1");
  dlo_plan* plan = new (std::nothrow) dlo_plan();
  if (!plan) DLO_FAIL(DLO_ERR_INVALID, "dlo_plan_create: out of host memory");
  plan->n_shards = n_shards;
  static std::atomic<uint64_t> next_id{1};
  plan->id = next_id.fetch_add(1);
  for (int32_t p = 0; p < n_params; ++p) {
    const dlo_param_desc& d = params[p];
    if (d.ndim < 1 || d.ndim > 4 || esize_of(d.dtype) == 0) {
      delete plan;
      DLO_FAIL(DLO_ERR_INVALID, "dlo_plan_create: param %d has ndim %d / dtype %d", p,
               d.ndim, d.dtype);
    }
    dlo_plan::Param q{};
    q.name = d.name ? d.name : "";
    q.ndim = d.ndim;
    q.dtype = d.dtype;
    q.numel = 1;
    for (int i = 0; i < 4; ++i) q.shape[i] = i < d.ndim ? d.shape[i] : 1;
    bool given = false;
    for (int i = 0; i < d.ndim; ++i) {
      if (d.shape[i] <= 0 || d.stride[i] < 0) {
        delete plan;
        DLO_FAIL(DLO_ERR_INVALID, "dlo_plan_create: param %d has extent %lld / stride %lld", p,
                 (long long)d.shape[i], (long long)d.stride[i]);
      }
      q.numel *= d.shape[i];
      given = given || d.stride[i] != 0;
    }
    // row-major strides of the logical shape
    int64_t rm[4] = {0, 0, 0, 0};
    for (int i = d.ndim - 1; i >= 0; --i) rm[i] = i == d.ndim - 1 ? 1 : rm[i + 1] * d.shape[i + 1];
    q.contiguous = true;
    q.storage_numel = 1;
    for (int i = 0; i < 4; ++i) q.stride[i] = 0;
    for (int i = 0; i < d.ndim; ++i) {
      q.stride[i] = given ? d.stride[i] : rm[i];
      q.storage_numel += (d.shape[i] - 1) * q.stride[i];
      if (d.shape[i] > 1 && q.stride[i] != rm[i]) q.contiguous = false;
    }
    // group by dtype, in order of first appearance
    int32_t g = -1;
    for (size_t i = 0; i < plan->groups.size(); ++i)
      if (plan->groups[i].dtype == d.dtype) g = static_cast<int32_t>(i);
    if (g < 0) {
      dlo_plan::Group grp{};
      grp.dtype = d.dtype;
      grp.esize = esize_of(d.dtype);
      plan->groups.push_back(grp);
      g = static_cast<int32_t>(plan->groups.size()) - 1;
    }
    q.group = g;
    q.group_offset = plan->groups[g].numel;
    plan->groups[g].numel += q.storage_numel;
    plan->params.push_back(q);
  }
  int64_t cursor = 0, stage_cursor = 0;
  for (auto& grp : plan->groups) {
    grp.shard_numel = (grp.numel + n_shards - 1) / n_shards;
    grp.shard_bytes = grp.shard_numel * grp.esize;
    grp.shard_alloc_bytes = round_up(grp.shard_bytes, 16);
    grp.base = round_up(cursor, kGroupAlign);
    cursor = grp.base + static_cast<int64_t>(n_shards) * grp.shard_bytes;
    // staging (DLO_COPY_STAGED): shard by shard, every shard 16-byte aligned
    grp.stage_base = round_up(stage_cursor, kGroupAlign);
    stage_cursor = grp.stage_base + static_cast<int64_t>(n_shards) * grp.shard_alloc_bytes;
  }
  plan->slot_bytes = cursor;
  plan->staging_bytes = stage_cursor;
  for (auto& q : plan->params)
    q.slot_offset = plan->groups[q.group].base + q.group_offset * plan->groups[q.group].esize;
  // DiT roles, by name; a role counts only with the dtype and the contiguous
  // layout the block forward reads
  bool all = true;
  for (int r = 0; r < R_COUNT; ++r) {
    plan->role[r] = -1;
    for (size_t p = 0; p < plan->params.size(); ++p) {
      const auto& q = plan->params[p];
      if (q.name == kRoleNames[r] && q.dtype == role_dtype(r) && q.contiguous)
        plan->role[r] = static_cast<int32_t>(p);
    }
    if (plan->role[r] < 0 && r < R_REQUIRED) all = false;
  }
  plan->has_dit_roles = all;
  *out = plan;
  clear_error();
  return DLO_OK;
}

dlo_status dlo_plan_query(const dlo_plan* plan, dlo_plan_info* out) {
  if (!plan || !out) DLO_FAIL(DLO_ERR_INVALID, "dlo_plan_query: null argument");
  out->n_params = static_cast<int32_t>(plan->params.size());
  out->n_groups = static_cast<int32_t>(plan->groups.size());
  out->n_shards = plan->n_shards;
  out->has_dit_roles = plan->has_dit_roles ? 1 : 0;
  out->slot_bytes = plan->slot_bytes;
  out->group_align = dlo::kGroupAlign;
  out->staging_bytes = plan->staging_bytes;
  return DLO_OK;
}

dlo_status dlo_plan_group(const dlo_plan* plan, int32_t group, dlo_group_info* out) {
  if (!plan || !out) DLO_FAIL(DLO_ERR_INVALID, "dlo_plan_group: null argument");
  if (group < 0 || group >= static_cast<int32_t>(plan->groups.size()))
    DLO_FAIL(DLO_ERR_INVALID, "dlo_plan_group: group %d out of range", group);
  const auto& g = plan->groups[group];
  out->dtype = g.dtype;
  out->esize = g.esize;
  out->numel = g.numel;
  out->shard_numel = g.shard_numel;
  out->shard_bytes = g.shard_bytes;
  out->shard_alloc_bytes = g.shard_alloc_bytes;
  out->base = g.base;
  out->stage_base = g.stage_base;
  return DLO_OK;
}

dlo_status dlo_plan_param(const dlo_plan* plan, int32_t param, dlo_param_info* out) {
  if (!plan || !out) DLO_FAIL(DLO_ERR_INVALID, "dlo_plan_param: null argument");
  if (param < 0 || param >= static_cast<int32_t>(plan->params.size()))
    DLO_FAIL(DLO_ERR_INVALID, "dlo_plan_param: param %d out of range", param);
  const auto& q = plan->params[param];
  out->group = q.group;
  out->dtype = q.dtype;
  out->numel = q.numel;
  out->group_offset = q.group_offset;
  out->slot_offset = q.slot_offset;
  out->storage_numel = q.storage_numel;
  for (int i = 0; i < 4; ++i) out->stride[i] = q.stride[i];
  return DLO_OK;
}

dlo_status dlo_shard_host(const dlo_plan* plan, const void* const* param_src,
                          void* const* shard_dst) {
  if (!plan || !param_src || !shard_dst)
    DLO_FAIL(DLO_ERR_INVALID, "dlo_shard_host: null argument");
  dlo::TraceRange range("shard_host", static_cast<int64_t>(plan->params.size()));
  const int32_t s = plan->n_shards;
  for (size_t g = 0; g < plan->groups.size(); ++g)
    for (int32_t r = 0; r < s; ++r)
      if (!shard_dst[g * s + r])
        DLO_FAIL(DLO_ERR_INVALID, "dlo_shard_host: shard (%zu,%d) is null", g, r);
  for (size_t p = 0; p < plan->params.size(); ++p)
    if (!param_src[p]) DLO_FAIL(DLO_ERR_INVALID, "dlo_shard_host: param %zu is null", p);
  for (size_t g = 0; g < plan->groups.size(); ++g) {
    const auto& grp = plan->groups[g];
    for (int32_t r = 0; r < s; ++r)
      std::memset(shard_dst[g * s + r], 0, static_cast<size_t>(grp.shard_alloc_bytes));
  }
  // Walk each parameter's elements in flat order and drop each contiguous
  // run into the shard whose window contains it.
  for (const auto& q : plan->params) {
    const auto& grp = plan->groups[q.group];
    const uint8_t* src = static_cast<const uint8_t*>(param_src[&q - plan->params.data()]);
    int64_t flat = q.group_offset;         // element index in the flat group
    int64_t left = q.storage_numel;        // storage extent, in memory order
    while (left > 0) {
      const int64_t r = flat / grp.shard_numel;
      const int64_t in_shard = flat - r * grp.shard_numel;
      const int64_t run = std::min(left, grp.shard_numel - in_shard);
      uint8_t* dst = static_cast<uint8_t*>(shard_dst[q.group * s + r]);
      std::memcpy(dst + in_shard * grp.esize, src, static_cast<size_t>(run * grp.esize));
      src += run * grp.esize;
      flat += run;
      left -= run;
    }
  }
  return DLO_OK;
}

dlo_status dlo_check_pieces(const dlo_plan* plan, int32_t phase, const dlo_copy_piece* pieces,
                            int32_t n, int64_t target_bytes, int32_t* bad) {
  if (bad) *bad = -1;
  if (!plan || n < 0 || (n > 0 && !pieces))
    DLO_FAIL(DLO_ERR_INVALID, "dlo_check_pieces: null argument or negative count");
  if (phase < DLO_PIECES_SLOT_FROM_SHARDS || phase > DLO_PIECES_SLOT_FROM_STAGING)
    DLO_FAIL(DLO_ERR_INVALID, "dlo_check_pieces: unknown phase %d", phase);
  const int32_t s = plan->n_shards;
  const int32_t n_groups = static_cast<int32_t>(plan->groups.size());
  const bool into_staging = phase == DLO_PIECES_STAGING_FROM_SHARDS;
  // per (group, shard): the byte ranges of the shard that some piece copies
  std::vector<std::vector<std::pair<int64_t, int64_t>>> covered(
      static_cast<size_t>(n_groups) * s);
  std::vector<std::pair<int64_t, int32_t>> by_dst;   // (dst_offset, piece)
  by_dst.reserve(static_cast<size_t>(n));
  for (int32_t i = 0; i < n; ++i) {
    const dlo_copy_piece& q = pieces[i];
    if (q.group < 0 || q.group >= n_groups || q.shard < 0 || q.shard >= s || q.bytes <= 0) {
      if (bad) *bad = i;
      DLO_FAIL(DLO_ERR_STATE, "dlo_check_pieces: piece %d names group %d / shard %d with %lld "
               "bytes (the plan has %d groups of %d shards)", i, q.group, q.shard,
               (long long)q.bytes, n_groups, s);
    }
    const auto& grp = plan->groups[q.group];
    const int64_t r = q.shard;
    const int64_t staged_at = grp.stage_base + r * grp.shard_alloc_bytes;
    const int64_t x = phase == DLO_PIECES_SLOT_FROM_STAGING ? q.src_offset - staged_at
                                                            : q.src_offset;
    const int64_t limit = into_staging ? grp.shard_alloc_bytes : grp.shard_bytes;
    if (x < 0 || x + q.bytes > limit) {
      if (bad) *bad = i;
      DLO_FAIL(DLO_ERR_STATE, "dlo_check_pieces: piece %d (group %d, shard %d) reads shard bytes "
               "[%lld, %lld) of %lld", i, q.group, q.shard, (long long)x,
               (long long)(x + q.bytes), (long long)limit);
    }
    const int64_t want = into_staging ? staged_at + x : grp.base + r * grp.shard_bytes + x;
    if (q.dst_offset != want) {
      if (bad) *bad = i;
      DLO_FAIL(DLO_ERR_STATE, "dlo_check_pieces: piece %d (group %d, shard %d) writes at byte "
               "%lld; those shard bytes belong at %lld", i, q.group, q.shard,
               (long long)q.dst_offset, (long long)want);
    }
    if (q.dst_offset < 0 || q.dst_offset + q.bytes > target_bytes) {
      if (bad) *bad = i;
      DLO_FAIL(DLO_ERR_STATE, "dlo_check_pieces: piece %d writes [%lld, %lld), past the "
               "target's %lld bytes", i, (long long)q.dst_offset,
               (long long)(q.dst_offset + q.bytes), (long long)target_bytes);
    }
    covered[static_cast<size_t>(q.group) * s + q.shard].push_back(
        {x, std::min(x + q.bytes, grp.shard_bytes)});
    by_dst.push_back({q.dst_offset, i});
  }
  std::sort(by_dst.begin(), by_dst.end());
  for (size_t j = 1; j < by_dst.size(); ++j) {
    const dlo_copy_piece& a = pieces[by_dst[j - 1].second];
    if (a.dst_offset + a.bytes > by_dst[j].first) {
      if (bad) *bad = by_dst[j].second;
      DLO_FAIL(DLO_ERR_STATE, "dlo_check_pieces: pieces %d and %d both write byte %lld",
               by_dst[j - 1].second, by_dst[j].second, (long long)by_dst[j].first);
    }
  }
  for (int32_t g = 0; g < n_groups; ++g)
    for (int32_t r = 0; r < s; ++r) {
      auto& iv = covered[static_cast<size_t>(g) * s + r];
      std::sort(iv.begin(), iv.end());
      int64_t end = 0;
      for (const auto& v : iv) {
        if (v.first > end) break;
        end = std::max(end, v.second);
      }
      if (end < plan->groups[g].shard_bytes)
        DLO_FAIL(DLO_ERR_STATE, "dlo_check_pieces: group %d shard %d: bytes from %lld of %lld "
                 "are not copied", g, r, (long long)end,
                 (long long)plan->groups[g].shard_bytes);
    }
  return DLO_OK;
}

void dlo_plan_destroy(dlo_plan* plan) { delete plan; }

}  // extern "C"
