// engine.cu — two device slots, the per-block hook schedule, and the
// prefetch (host->device copy plus reassembly) on a dedicated copy stream.
//
// "Distributed Layerwise Offload" (vLLM blog preview, 2026-07-30):
//   "Weight Sharding + AllGather": H2D of each shard on copy_stream, gather
//     of the full block, re-pointing of parameters, forward on a compute
//     stream that waits for the gather event; block N+1's preparation
//     overlaps block N's forward.
//   "Double-Buffer Memory Bound": exactly two blocks on the device.
//   "Slot Tracking: i%2 + Dynamic Correction": hook i starts at slot i % 2;
//     when the previous hook has prefetched, the hook takes that slot, which
//     keeps the circular tail->head prefetch of an odd block count from
//     landing in the slot the head reads.
// "Distributed Layerwise Offload: Scaling Toward 200B+ DiT Models
// Efficiently in vLLM-Omni", "3. Double-Buffered Prefetch with H2D +
// AllGather Overlap": two buffers sized to the largest block, shared by all
// blocks, event-based synchronisation between streams.
//
// Beyond the pages: the prefetch into a slot also waits for the free event
// recorded after the last forward that read that slot (the pages draw only
// the compute-waits-for-gather arrow; reusing two buffers needs the reverse
// write-after-read wait too).
#include <algorithm>
#include <chrono>
#include <condition_variable>
#include <cstring>
#include <mutex>
#include <new>
#include <thread>

#include "common.h"
#include "trace.h"

namespace dlo {
dlo_status forward_impl(const dlo_dit_cfg* cfg, const dlo_plan* plan, const void* block_base,
                        float* x, void* scratch, size_t scratch_bytes, cudaStream_t stream);
}

namespace dlo {

// CPU threads that pack a rank-local block: run() hands the copy tasks to
// the pool's threads and the calling thread and returns once all are done.
class PackPool {
 public:
  struct Task {
    uint8_t* dst;
    const uint8_t* src;
    size_t n;
  };
  explicit PackPool(int threads) {
    for (int i = 1; i < threads; ++i) th_.emplace_back([this] { loop(); });
  }
  ~PackPool() {
    {
      std::lock_guard<std::mutex> l(mu_);
      stop_ = true;
    }
    cv_.notify_all();
    for (auto& t : th_) t.join();
  }
  void run(const std::vector<Task>& tasks) {
    {
      std::lock_guard<std::mutex> l(mu_);
      tasks_ = &tasks;
      next_ = 0;
      left_ = tasks.size();
      ++gen_;
    }
    cv_.notify_all();
    work();
    std::unique_lock<std::mutex> l(mu_);
    done_.wait(l, [this] { return left_ == 0; });
    tasks_ = nullptr;
  }

 private:
  void work() {
    for (;;) {
      const Task* t;
      {
        std::lock_guard<std::mutex> l(mu_);
        if (!tasks_ || next_ >= tasks_->size()) return;
        t = &(*tasks_)[next_++];
      }
      std::memcpy(t->dst, t->src, t->n);
      std::lock_guard<std::mutex> l(mu_);
      if (--left_ == 0) done_.notify_all();
    }
  }
  void loop() {
    uint64_t seen = 0;
    for (;;) {
      {
        std::unique_lock<std::mutex> l(mu_);
        cv_.wait(l, [&] { return stop_ || (gen_ != seen && tasks_ && next_ < tasks_->size()); });
        if (stop_) return;
        seen = gen_;
      }
      work();
    }
  }
  std::vector<std::thread> th_;
  std::mutex mu_;
  std::condition_variable cv_, done_;
  const std::vector<Task>* tasks_ = nullptr;
  size_t next_ = 0, left_ = 0;
  uint64_t gen_ = 0;
  bool stop_ = false;
};

// Fixed-capacity ring: grows to `cap` entries, then each push overwrites
// the oldest one (counted in `dropped`).  at(0) is the oldest entry kept.
template <class T>
class Ring {
 public:
  void set_capacity(size_t cap) { cap_ = cap; }
  // The entry to fill next; *reused = true when it is an evicted old entry
  // (its fields still hold that entry's values).
  T& push(bool* reused) {
    if (buf_.size() < cap_) {
      buf_.emplace_back();
      *reused = false;
      return buf_.back();
    }
    T& t = buf_[head_];
    head_ = (head_ + 1) % cap_;
    ++dropped_;
    *reused = true;
    return t;
  }
  size_t size() const { return buf_.size(); }
  const T& at(size_t i) const { return buf_.size() < cap_ ? buf_[i] : buf_[(head_ + i) % cap_]; }
  int64_t dropped() const { return dropped_; }
  // every stored entry, in storage order (for releasing resources)
  const std::vector<T>& storage() const { return buf_; }

 private:
  std::vector<T> buf_;
  size_t cap_ = 0, head_ = 0;
  int64_t dropped_ = 0;
};

}  // namespace dlo

struct dlo_engine {
  struct Block {
    const dlo_plan* plan = nullptr;
    std::vector<const void*> host;   // [g * n_shards + r]
    std::vector<const void*> dev;    // device-accessible addresses (null: DMA only)
    std::vector<int64_t> pitch;      // [g]: constant host stride between shards, 0 if none
    int64_t bytes = 0;               // bytes one prefetch moves
    // rank-local source block (dlo_register_block_source): parameters by
    // address; direct = every one page-locked (copied straight into the slot)
    struct Src {
      const uint8_t* p;
      int64_t bytes;
      int64_t off;                   // byte offset in a slot
    };
    bool source = false;
    bool direct = false;
    std::vector<Src> src;
  };
  struct Hook {
    int32_t current_slot;
    int32_t prefetched_slot;         // -1: none yet
  };
  struct Timed {
    cudaEvent_t a, b;
    int64_t bytes;
    int32_t mode;
    int64_t seq;                     // n-th timed prefetch of the engine
    int32_t block, slot;
  };
  static constexpr int kMaxFan = 8;

  int32_t n_blocks = 0;
  uint8_t* slot[2] = {nullptr, nullptr};
  int64_t slot_bytes = 0;
  cudaStream_t compute = nullptr, copy = nullptr;
  // prefetches into slot x run on slot_copy[x]: the caller's copy stream,
  // or for slot 1 a library-owned one with two_copy_streams, so that
  // consecutive block copies may overlap at their ends
  cudaStream_t slot_copy[2] = {nullptr, nullptr};
  cudaStream_t own_copy = nullptr;
  int32_t mode = DLO_COPY_AUTO;
  int32_t copy_ctas = 0;
  bool timing = false;
  bool poison = false;               // debugging: 0xA5 over each slot after its forward
  bool checks = false;               // debugging: offsets of every copy checked before issue
  int64_t checked_pieces = 0;
  std::vector<Block> blocks;
  std::vector<Hook> hooks;
  cudaEvent_t ready[2] = {nullptr, nullptr};
  cudaEvent_t freed[2] = {nullptr, nullptr};
  int32_t slot_holds[2] = {-1, -1};
  int32_t last_reader[2] = {-1, -1};
  int64_t k = 0;                     // next global forward index
  bool in_forward = false;
  int32_t cur_block = -1, cur_slot = -1;
  int64_t fill_seq[2] = {-1, -1};    // prefetch count when each slot was last filled
  // the newest entries only: one per forward, and (timing = 1) one per
  // prefetch; a full ring overwrites its oldest entry and counts it dropped
  dlo::Ring<dlo_sched_event> log;
  dlo::Ring<Timed> timed;
  // DMA fan-out (library-owned streams forked from / joined to `copy`)
  int32_t fan = 1;
  cudaStream_t aux[kMaxFan] = {};
  cudaEvent_t fork_ev = nullptr;
  cudaEvent_t join_ev[kMaxFan] = {};
  // DMA mode: dtype groups smaller than kSmallGroupBytes move by a one-CTA
  // copy-kernel launch on this side stream, concurrent with the large DMA
  cudaStream_t side = nullptr;
  cudaEvent_t side_fork = nullptr, side_join = nullptr;
  // AUTO race: timing events on the compute stream at the window edges
  // (windows DMA, kernel, DMA, kernel; two events each)
  cudaEvent_t race_ev[8] = {};
  bool race_rec[8] = {false, false, false, false, false, false, false, false};
  int32_t chosen = -1;               // DLO_COPY_DMA / DLO_COPY_KERNEL once decided
  // DLO_COPY_STAGED: caller-owned staging buffers (staging[x] serves slot x)
  // and gather stream; staged[x] marks the H2D into staging[x] done,
  // stage_free[x] the gather out of it
  uint8_t* staging[2] = {nullptr, nullptr};
  int64_t staging_bytes = 0;
  cudaStream_t gather = nullptr;
  cudaEvent_t staged[2] = {nullptr, nullptr};
  cudaEvent_t stage_free[2] = {nullptr, nullptr};
  // rank-local source blocks: caller-owned pinned host staging (host staging
  // x serves slot x), the event of the last DMA out of each, the CPU pool
  // that packs, and counters
  uint8_t* host_staging[2] = {nullptr, nullptr};
  int64_t host_staging_bytes = 0;
  cudaEvent_t hs_read[2] = {nullptr, nullptr};
  bool hs_pending[2] = {false, false};
  dlo::PackPool* pool = nullptr;
  int64_t n_direct = 0, n_packed = 0;
  int64_t n_copy_launches = 0;
  double pack_ms = 0;
  double race_dma_us = 0, race_kernel_us = 0;
  int64_t n_prefetches = 0;
  int64_t n_kernel_prefetches = 0;
  int64_t n_timed = 0;               // timed prefetches so far (next seq)
};

namespace dlo {
dlo_status preload_kernels();
namespace {

// AUTO races DMA against the copy kernel on the compute stream's time per
// forward.  Four windows of W forwards follow s = race_start(n_blocks):
// the prefetches issued by the forwards of windows 0 and 2 use DMA, those
// of windows 1 and 3 the copy kernel.  Forward k+1 reads what the prefetch
// issued at forward k brought in and overlaps the prefetch issued at k+1,
// so the free-event intervals inside a window see only that window's mode.
// Each mode keeps its better window, which discounts a one-off stall.
// The race starts after one full pass over the blocks plus two forwards,
// so that one-time costs (module loading, first launches, the first
// device access to each pinned host page) stay out of every window.
constexpr int64_t kRaceWindow = 6;
constexpr int32_t kDefaultLogCapacity = 65536;
constexpr int kRaceWindows = 4;
inline int64_t race_start(int32_t n_blocks) { return static_cast<int64_t>(n_blocks) + 2; }

// With desc.checks, a prefetch's copies are first listed here by offsets
// (into `target`, from each piece's own shard or from staging) instead of
// issued, and checked against the plan with dlo_check_pieces.
struct DryRun {
  std::vector<dlo_copy_piece> pieces;
  const uint8_t* target = nullptr;
  void add(int32_t g, int32_t r, const void* dst, const void* src, const void* src_base,
           int64_t bytes) {
    dlo_copy_piece q;
    q.group = g;
    q.shard = r;
    q.dst_offset = static_cast<const uint8_t*>(dst) - target;
    q.src_offset = static_cast<const uint8_t*>(src) - static_cast<const uint8_t*>(src_base);
    q.bytes = bytes;
    pieces.push_back(q);
  }
};

dlo_status build_segments(const dlo_engine::Block& b, uint8_t* dst, SegmentTable* t) {
  const dlo_plan* p = b.plan;
  const int32_t s = p->n_shards;
  t->n = 0;
  for (size_t g = 0; g < p->groups.size(); ++g) {
    const auto& grp = p->groups[g];
    for (int32_t r = 0; r < s; ++r) {
      if (t->n >= kMaxSegments)
        DLO_FAIL(DLO_ERR_INVALID, "prefetch: more than %d (group, shard) pieces", kMaxSegments);
      Segment& sg = t->seg[t->n++];
      sg.src = b.dev[g * s + r];
      sg.dst = dst + grp.base + static_cast<int64_t>(r) * grp.shard_bytes;
      sg.bytes = grp.shard_bytes;
    }
  }
  return DLO_OK;
}

// A group whose shards sit at a constant host stride (>= the shard bytes)
// can move as one 2-D DMA: rows = shards, row width = shard bytes, source
// pitch = the stride, destination pitch = the shard bytes (the gathered
// layout).  Returns that stride, or 0.
void compute_pitches(dlo_engine::Block* b) {
  const dlo_plan* p = b->plan;
  const int32_t s = p->n_shards;
  b->pitch.assign(p->groups.size(), 0);
  for (size_t g = 0; g < p->groups.size(); ++g) {
    if (s < 2) continue;
    const char* h0 = static_cast<const char*>(b->host[g * s]);
    const int64_t stride = static_cast<const char*>(b->host[g * s + 1]) - h0;
    bool ok = stride >= p->groups[g].shard_bytes;
    for (int32_t r = 2; ok && r < s; ++r)
      ok = static_cast<const char*>(b->host[g * s + r]) - h0 == stride * r;
    if (ok) b->pitch[g] = stride;
  }
}

bool all_mapped(const dlo_engine::Block& b) {
  for (const void* q : b.dev)
    if (!q) return false;
  return true;
}

// One prefetch's bytes: the copy kernel (one launch), or DMA — one
// cudaMemcpyAsync per (group, shard) to its final slot offset, dealt to up
// to `fan` streams (largest first, each to the least-loaded stream) that
// fork from `stream` and join back into it.
// Small groups (the f32 norm/adaLN vectors: a few tens of KB) pay more for
// a DMA's setup than for their bytes; they go by copy kernel on a side
// stream while the large group's DMA runs.
constexpr int64_t kSmallGroupBytes = 1 << 20;

dlo_status copy_block(const dlo_engine::Block& b, uint8_t* dst, int32_t mode, int ctas,
                      cudaStream_t stream, int fan, cudaStream_t* aux, cudaEvent_t fork_ev,
                      cudaEvent_t* join_ev, cudaStream_t side = nullptr,
                      cudaEvent_t side_fork = nullptr, cudaEvent_t side_join = nullptr,
                      int64_t* launches = nullptr, DryRun* dry = nullptr) {
  const dlo_plan* p = b.plan;
  const int32_t s = p->n_shards;
  if (mode == DLO_COPY_KERNEL) {
    if (!all_mapped(b))
      DLO_FAIL(DLO_ERR_INVALID, "prefetch: a shard is not device-mapped pinned memory");
    SegmentTable t;
    DLO_TRY(build_segments(b, dst, &t));
    if (dry) {
      for (int32_t i = 0; i < t.n; ++i)
        dry->add(i / s, i % s, t.seg[i].dst, t.seg[i].src, b.dev[i], t.seg[i].bytes);
      return DLO_OK;
    }
    if (launches) ++*launches;
    return launch_copy_reassemble(t, ctas, stream);
  }
  std::vector<char> by_kernel(p->groups.size(), 0);
  if (side && all_mapped(b) && p->groups.size() > 1) {
    SegmentTable t;
    t.n = 0;
    for (size_t g = 0; g < p->groups.size(); ++g) {
      const auto& grp = p->groups[g];
      if (grp.shard_bytes * s >= kSmallGroupBytes || t.n + s > kMaxSegments) continue;
      by_kernel[g] = 1;
      for (int32_t r = 0; r < s; ++r) {
        Segment& sg = t.seg[t.n++];
        sg.src = b.dev[g * s + r];
        sg.dst = dst + grp.base + static_cast<int64_t>(r) * grp.shard_bytes;
        sg.bytes = grp.shard_bytes;
        if (dry) dry->add(static_cast<int32_t>(g), r, sg.dst, sg.src, b.dev[g * s + r], sg.bytes);
      }
    }
    if (t.n > 0 && !dry) {
      DLO_CUDA(cudaEventRecord(side_fork, stream));
      DLO_CUDA(cudaStreamWaitEvent(side, side_fork, 0));
      DLO_TRY(launch_copy_reassemble(t, 1, side));
      if (launches) ++*launches;
      DLO_CUDA(cudaEventRecord(side_join, side));
    }
  }
  struct Piece { uint8_t* dst; const void* src; int64_t bytes; };
  std::vector<Piece> pieces;
  for (size_t g = 0; g < p->groups.size(); ++g) {
    const auto& grp = p->groups[g];
    if (by_kernel[g]) continue;
    if (fan <= 1 && !b.pitch.empty() && b.pitch[g] > 0) {
      if (dry) {
        // a linear copy (pitch = shard bytes) or a 2-D copy: row r of it
        for (int32_t r = 0; r < s; ++r)
          dry->add(static_cast<int32_t>(g), r,
                   dst + grp.base + static_cast<int64_t>(r) * grp.shard_bytes,
                   static_cast<const uint8_t*>(b.host[g * s]) + r * b.pitch[g],
                   b.host[g * s + r], grp.shard_bytes);
        continue;
      }
      if (b.pitch[g] == grp.shard_bytes) {
        // the shards are back to back in host memory: one linear copy
        DLO_CUDA(cudaMemcpyAsync(dst + grp.base, b.host[g * s],
                                 static_cast<size_t>(grp.shard_bytes) * s,
                                 cudaMemcpyHostToDevice, stream));
      } else {
        // all shards of the group in one 2-D copy
        DLO_CUDA(cudaMemcpy2DAsync(dst + grp.base, static_cast<size_t>(grp.shard_bytes),
                                   b.host[g * s], static_cast<size_t>(b.pitch[g]),
                                   static_cast<size_t>(grp.shard_bytes), static_cast<size_t>(s),
                                   cudaMemcpyHostToDevice, stream));
      }
      continue;
    }
    for (int32_t r = 0; r < s; ++r) {
      pieces.push_back({dst + grp.base + static_cast<int64_t>(r) * grp.shard_bytes,
                        b.host[g * s + r], grp.shard_bytes});
      if (dry)
        dry->add(static_cast<int32_t>(g), r, pieces.back().dst, pieces.back().src,
                 b.host[g * s + r], grp.shard_bytes);
    }
  }
  if (dry) return DLO_OK;
  auto join_side = [&]() -> dlo_status {
    for (size_t g = 0; g < by_kernel.size(); ++g)
      if (by_kernel[g]) {
        DLO_CUDA(cudaStreamWaitEvent(stream, side_join, 0));
        break;
      }
    return DLO_OK;
  };
  if (pieces.empty()) return join_side();
  const int used = static_cast<int>(std::min<size_t>(fan, pieces.size()));
  if (used <= 1) {
    for (const Piece& q : pieces)
      DLO_CUDA(cudaMemcpyAsync(q.dst, q.src, static_cast<size_t>(q.bytes),
                               cudaMemcpyHostToDevice, stream));
    return join_side();
  }
  std::stable_sort(pieces.begin(), pieces.end(),
                   [](const Piece& a, const Piece& c) { return a.bytes > c.bytes; });
  std::vector<int64_t> load(used, 0);
  DLO_CUDA(cudaEventRecord(fork_ev, stream));
  for (int j = 0; j < used; ++j) DLO_CUDA(cudaStreamWaitEvent(aux[j], fork_ev, 0));
  for (const Piece& q : pieces) {
    int j = 0;
    for (int c = 1; c < used; ++c)
      if (load[c] < load[j]) j = c;
    load[j] += q.bytes;
    DLO_CUDA(cudaMemcpyAsync(q.dst, q.src, static_cast<size_t>(q.bytes),
                             cudaMemcpyHostToDevice, aux[j]));
  }
  for (int j = 0; j < used; ++j) {
    DLO_CUDA(cudaEventRecord(join_ev[j], aux[j]));
    DLO_CUDA(cudaStreamWaitEvent(stream, join_ev[j], 0));
  }
  return join_side();
}

// DLO_COPY_STAGED, phase 1 (the H2D of [B2] §3): every shard host->device
// by DMA into the staging buffer, shard by shard — group g, shard r at
// stage_base_g + r * shard_alloc_bytes (16-byte aligned).  A group whose
// host shards sit at a constant stride moves as one 2-D copy (one linear
// copy when that stride equals the staging stride).
dlo_status stage_h2d(const dlo_engine::Block& b, uint8_t* staging, cudaStream_t stream,
                     DryRun* dry = nullptr) {
  const dlo_plan* p = b.plan;
  const int32_t s = p->n_shards;
  for (size_t g = 0; g < p->groups.size(); ++g) {
    const auto& grp = p->groups[g];
    uint8_t* d0 = staging + grp.stage_base;
    const int64_t sp = grp.shard_alloc_bytes;
    const int64_t hp = b.pitch.empty() ? 0 : b.pitch[g];
    if (dry) {
      // row r of the linear (hp = sp) or 2-D copy, or the per-shard copy
      const uint8_t* h0 = static_cast<const uint8_t*>(b.host[g * s]);
      for (int32_t r = 0; r < s; ++r)
        dry->add(static_cast<int32_t>(g), r, d0 + r * sp,
                 hp > 0 ? h0 + r * hp : b.host[g * s + r], b.host[g * s + r],
                 hp == sp ? sp : grp.shard_bytes);
      continue;
    }
    if (hp == sp) {
      DLO_CUDA(cudaMemcpyAsync(d0, b.host[g * s], static_cast<size_t>(sp) * s,
                               cudaMemcpyHostToDevice, stream));
    } else if (hp > 0) {
      DLO_CUDA(cudaMemcpy2DAsync(d0, static_cast<size_t>(sp), b.host[g * s],
                                 static_cast<size_t>(hp), static_cast<size_t>(grp.shard_bytes),
                                 static_cast<size_t>(s), cudaMemcpyHostToDevice, stream));
    } else {
      for (int32_t r = 0; r < s; ++r)
        DLO_CUDA(cudaMemcpyAsync(d0 + static_cast<int64_t>(r) * sp, b.host[g * s + r],
                                 static_cast<size_t>(grp.shard_bytes), cudaMemcpyHostToDevice,
                                 stream));
    }
  }
  return DLO_OK;
}

// DLO_COPY_STAGED, phase 2 (the AllGather of [B2] §3 on one device): the
// copy-and-reassemble kernel moves every staged shard to its slot offset
// (group base + r * shard_bytes), i.e. the concatenation in rank order that
// all_gather_into_tensor produces.
dlo_status stage_gather(const dlo_plan* p, const uint8_t* staging, uint8_t* dst, int ctas,
                        cudaStream_t stream, DryRun* dry = nullptr) {
  const int32_t s = p->n_shards;
  SegmentTable t;
  t.n = 0;
  for (size_t g = 0; g < p->groups.size(); ++g) {
    const auto& grp = p->groups[g];
    for (int32_t r = 0; r < s; ++r) {
      if (t.n >= kMaxSegments)
        DLO_FAIL(DLO_ERR_INVALID, "staged gather: more than %d (group, shard) pieces",
                 kMaxSegments);
      Segment& sg = t.seg[t.n++];
      sg.src = staging + grp.stage_base + static_cast<int64_t>(r) * grp.shard_alloc_bytes;
      sg.dst = dst + grp.base + static_cast<int64_t>(r) * grp.shard_bytes;
      sg.bytes = grp.shard_bytes;
      if (dry) dry->add(static_cast<int32_t>(g), r, sg.dst, sg.src, staging, sg.bytes);
    }
  }
  if (dry) return DLO_OK;
  return launch_copy_reassemble(t, ctas, stream);
}

// AUTO: decide once the four window-edge events have completed
// (non-blocking).
void try_decide(dlo_engine* e) {
  if (e->chosen >= 0) return;
  for (int i = 0; i < 2 * kRaceWindows; ++i)
    if (!e->race_rec[i] || cudaEventQuery(e->race_ev[i]) != cudaSuccess) return;
  double best[2] = {1e30, 1e30};   // [0] DMA, [1] kernel
  for (int w = 0; w < kRaceWindows; ++w) {
    float ms = 0;
    if (cudaEventElapsedTime(&ms, e->race_ev[2 * w], e->race_ev[2 * w + 1]) != cudaSuccess) {
      // no measurement: no choice can rest on it, so DMA (which takes no
      // SM time from the forward) is kept; -1 marks the race unmeasured
      cudaGetLastError();
      e->race_dma_us = e->race_kernel_us = -1.0;
      e->chosen = DLO_COPY_DMA;
      return;
    }
    const double us = 1e3 * ms / (kRaceWindow - 1);
    best[w & 1] = std::min(best[w & 1], us);
  }
  e->race_dma_us = best[0];
  e->race_kernel_us = best[1];
  e->chosen = e->race_kernel_us < e->race_dma_us ? DLO_COPY_KERNEL : DLO_COPY_DMA;
}

// Mode of a prefetch issued by forward k (k < 0: outside the hook).
int32_t mode_for(dlo_engine* e, int64_t k, const dlo_engine::Block& b) {
  if (e->mode != DLO_COPY_AUTO) return e->mode;
  try_decide(e);
  if (e->chosen >= 0) return e->chosen;
  const int64_t s0 = race_start(e->n_blocks);
  const int64_t w = k >= s0 ? (k - s0) / kRaceWindow : -1;
  if (w >= 0 && w < kRaceWindows && (w & 1)) {
    if (!all_mapped(b)) {   // the kernel cannot read this block: no race
      e->chosen = DLO_COPY_DMA;
      return DLO_COPY_DMA;
    }
    return DLO_COPY_KERNEL;
  }
  return DLO_COPY_DMA;
}

// The timing entry of the prefetch about to be enqueued: a new entry with
// two new events, or (ring full) the oldest entry, whose events are
// recorded again.
dlo_status timed_entry(dlo_engine* e, int64_t bytes, int32_t mode, int32_t block, int32_t slot,
                       dlo_engine::Timed** out) {
  bool reused = false;
  dlo_engine::Timed& t = e->timed.push(&reused);
  if (!reused) {
    t.a = t.b = nullptr;
    if (cudaEventCreate(&t.a) != cudaSuccess || cudaEventCreate(&t.b) != cudaSuccess) {
      cudaGetLastError();
      DLO_FAIL(DLO_ERR_CUDA, "cudaEventCreate failed");
    }
  }
  t.bytes = bytes;
  t.mode = mode;
  t.seq = e->n_timed++;
  t.block = block;
  t.slot = slot;
  *out = &t;
  return DLO_OK;
}

// Bookkeeping of a prefetch just enqueued into `slot`.
void mark_filled(dlo_engine* e, int32_t slot, int32_t block) {
  e->slot_holds[slot] = block;
  e->fill_seq[slot] = e->n_prefetches;
  e->n_prefetches++;
}

// Host-side bounded wait for an event (polls; false after timeout_ms).
bool wait_event_host(cudaEvent_t ev, int timeout_ms) {
  const auto t0 = std::chrono::steady_clock::now();
  for (;;) {
    const cudaError_t q = cudaEventQuery(ev);
    if (q == cudaSuccess) return true;
    if (q != cudaErrorNotReady) return false;
    if (std::chrono::steady_clock::now() - t0 > std::chrono::milliseconds(timeout_ms))
      return false;
    std::this_thread::sleep_for(std::chrono::microseconds(20));
  }
}

constexpr int kHostStagingWaitMs = 60000;

// Prefetch of a rank-local source block into `slot` ([D5] "Rank-local path
// without DLO AllGather").  Direct: every parameter copied by DMA from its
// page-locked source to its slot offset.  Packed: once the DMA that last
// read host staging `slot` is done, CPU threads copy the parameters to
// their slot offsets inside it, then one DMA moves the packed block.
dlo_status prefetch_source(dlo_engine* e, int32_t block, int32_t slot) {
  const dlo_engine::Block& b = e->blocks[block];
  cudaStream_t cs = e->slot_copy[slot];
  dlo_engine::Timed* t = nullptr;
  if (e->timing) DLO_TRY(timed_entry(e, b.bytes, DLO_COPY_DMA, block, slot, &t));
  if (b.direct) {
    DLO_CUDA(cudaStreamWaitEvent(cs, e->freed[slot], 0));
    if (t) DLO_CUDA(cudaEventRecord(t->a, cs));
    for (const auto& s : b.src)
      DLO_CUDA(cudaMemcpyAsync(e->slot[slot] + s.off, s.p, static_cast<size_t>(s.bytes),
                               cudaMemcpyHostToDevice, cs));
    e->n_direct++;
  } else {
    const auto t0 = std::chrono::steady_clock::now();
    if (e->hs_pending[slot] && !wait_event_host(e->hs_read[slot], kHostStagingWaitMs))
      DLO_FAIL(DLO_ERR_TIMEOUT, "prefetch: host staging %d not released by its DMA", slot);
    std::vector<PackPool::Task> tasks;
    constexpr size_t kPiece = 4u << 20;
    for (const auto& s : b.src)
      for (int64_t o = 0; o < s.bytes; o += static_cast<int64_t>(kPiece))
        tasks.push_back({e->host_staging[slot] + s.off + o, s.p + o,
                         static_cast<size_t>(std::min<int64_t>(kPiece, s.bytes - o))});
    {
      TraceRange pack("pack", block);
      e->pool->run(tasks);
    }
    e->pack_ms += std::chrono::duration<double, std::milli>(std::chrono::steady_clock::now() - t0)
                      .count();
    DLO_CUDA(cudaStreamWaitEvent(cs, e->freed[slot], 0));
    if (t) DLO_CUDA(cudaEventRecord(t->a, cs));
    DLO_CUDA(cudaMemcpyAsync(e->slot[slot], e->host_staging[slot],
                             static_cast<size_t>(b.plan->slot_bytes), cudaMemcpyHostToDevice,
                             cs));
    DLO_CUDA(cudaEventRecord(e->hs_read[slot], cs));
    e->hs_pending[slot] = true;
    e->n_packed++;
  }
  if (t) DLO_CUDA(cudaEventRecord(t->b, cs));
  DLO_CUDA(cudaEventRecord(e->ready[slot], cs));
  mark_filled(e, slot, block);
  return DLO_OK;
}

// desc.checks: lists the copies a prefetch of `b` into `slot` in `mode`
// would issue (nothing is issued) and checks their offsets against the
// plan; the prefetch is refused if one fails.
dlo_status check_prefetch(dlo_engine* e, const dlo_engine::Block& b, int32_t slot,
                          int32_t mode) {
  int32_t bad = -1;
  if (mode == DLO_COPY_STAGED) {
    DryRun h2d, gather;
    h2d.target = e->staging[slot];
    gather.target = e->slot[slot];
    DLO_TRY(stage_h2d(b, e->staging[slot], nullptr, &h2d));
    DLO_TRY(stage_gather(b.plan, e->staging[slot], e->slot[slot], 0, nullptr, &gather));
    DLO_TRY(dlo_check_pieces(b.plan, DLO_PIECES_STAGING_FROM_SHARDS, h2d.pieces.data(),
                             static_cast<int32_t>(h2d.pieces.size()), e->staging_bytes, &bad));
    DLO_TRY(dlo_check_pieces(b.plan, DLO_PIECES_SLOT_FROM_STAGING, gather.pieces.data(),
                             static_cast<int32_t>(gather.pieces.size()), e->slot_bytes, &bad));
    e->checked_pieces += static_cast<int64_t>(h2d.pieces.size() + gather.pieces.size());
    return DLO_OK;
  }
  DryRun d;
  d.target = e->slot[slot];
  DLO_TRY(copy_block(b, e->slot[slot], mode, e->copy_ctas, nullptr, e->fan, e->aux, e->fork_ev,
                     e->join_ev, e->side, e->side_fork, e->side_join, nullptr, &d));
  DLO_TRY(dlo_check_pieces(b.plan, DLO_PIECES_SLOT_FROM_SHARDS, d.pieces.data(),
                           static_cast<int32_t>(d.pieces.size()), e->slot_bytes, &bad));
  e->checked_pieces += static_cast<int64_t>(d.pieces.size());
  return DLO_OK;
}

// Enqueues the prefetch of `block` into `slot` on the copy stream.
dlo_status enqueue_prefetch(dlo_engine* e, int32_t block, int32_t slot, int64_t issued_by_k,
                            int32_t* used_mode = nullptr) {
  TraceRange range(slot ? "prefetch slot 1" : "prefetch slot 0", block);
  const dlo_engine::Block& b = e->blocks[block];
  cudaStream_t cs = e->slot_copy[slot];
  if (b.source) {
    if (used_mode) *used_mode = DLO_COPY_DMA;
    return prefetch_source(e, block, slot);
  }
  const int32_t mode = mode_for(e, issued_by_k, b);
  if (used_mode) *used_mode = mode;
  if (e->checks) DLO_TRY(check_prefetch(e, b, slot, mode));
  if (mode == DLO_COPY_STAGED) {
    // H2D into staging[slot] once the gather that last read it is done;
    // the gather then waits for the H2D and for the slot's free event
    DLO_CUDA(cudaStreamWaitEvent(cs, e->stage_free[slot], 0));
    dlo_engine::Timed* t = nullptr;
    if (e->timing) {
      DLO_TRY(timed_entry(e, b.bytes, mode, block, slot, &t));
      DLO_CUDA(cudaEventRecord(t->a, cs));
    }
    DLO_TRY(stage_h2d(b, e->staging[slot], cs));
    if (t) DLO_CUDA(cudaEventRecord(t->b, cs));
    DLO_CUDA(cudaEventRecord(e->staged[slot], cs));
    DLO_CUDA(cudaStreamWaitEvent(e->gather, e->staged[slot], 0));
    DLO_CUDA(cudaStreamWaitEvent(e->gather, e->freed[slot], 0));
    DLO_TRY(stage_gather(b.plan, e->staging[slot], e->slot[slot], e->copy_ctas, e->gather));
    e->n_copy_launches++;
    DLO_CUDA(cudaEventRecord(e->stage_free[slot], e->gather));
    DLO_CUDA(cudaEventRecord(e->ready[slot], e->gather));
    mark_filled(e, slot, block);
    return DLO_OK;
  }
  DLO_CUDA(cudaStreamWaitEvent(cs, e->freed[slot], 0));
  dlo_engine::Timed* t = nullptr;
  if (e->timing) {
    DLO_TRY(timed_entry(e, b.bytes, mode, block, slot, &t));
    DLO_CUDA(cudaEventRecord(t->a, cs));
  }
  DLO_TRY(copy_block(b, e->slot[slot], mode, e->copy_ctas, cs, e->fan, e->aux, e->fork_ev,
                     e->join_ev, e->side, e->side_fork, e->side_join, &e->n_copy_launches));
  if (t) DLO_CUDA(cudaEventRecord(t->b, cs));
  DLO_CUDA(cudaEventRecord(e->ready[slot], cs));
  mark_filled(e, slot, block);
  if (mode == DLO_COPY_KERNEL) e->n_kernel_prefetches++;
  return DLO_OK;
}

dlo_status check_engine(const dlo_engine* e) {
  if (!e) DLO_FAIL(DLO_ERR_INVALID, "null engine");
  return DLO_OK;
}

// The slot whose copy of `block` a forward reads: during that block's
// forward, the slot the hook picked; otherwise the slot filled with it last
// (both slots hold the same block when the pass has one block: the newer
// copy is the one the next forward reads).
int32_t slot_of(const dlo_engine* e, int32_t block) {
  if (e->in_forward && block == e->cur_block) return e->cur_slot;
  const bool h0 = e->slot_holds[0] == block, h1 = e->slot_holds[1] == block;
  if (h0 && h1) return e->fill_seq[1] > e->fill_seq[0] ? 1 : 0;
  if (h0) return 0;
  if (h1) return 1;
  return -1;
}

void release(dlo_engine* e) {
  for (int s = 0; s < 2; ++s) {
    if (e->ready[s]) cudaEventDestroy(e->ready[s]);
    if (e->freed[s]) cudaEventDestroy(e->freed[s]);
    if (e->staged[s]) cudaEventDestroy(e->staged[s]);
    if (e->stage_free[s]) cudaEventDestroy(e->stage_free[s]);
    if (e->hs_read[s]) cudaEventDestroy(e->hs_read[s]);
  }
  delete e->pool;
  if (e->own_copy) cudaStreamDestroy(e->own_copy);
  for (const auto& t : e->timed.storage()) {
    if (t.a) cudaEventDestroy(t.a);
    if (t.b) cudaEventDestroy(t.b);
  }
  for (int i = 0; i < 8; ++i)
    if (e->race_ev[i]) cudaEventDestroy(e->race_ev[i]);
  if (e->fork_ev) cudaEventDestroy(e->fork_ev);
  if (e->side_fork) cudaEventDestroy(e->side_fork);
  if (e->side_join) cudaEventDestroy(e->side_join);
  if (e->side) cudaStreamDestroy(e->side);
  for (int j = 0; j < dlo_engine::kMaxFan; ++j) {
    if (e->join_ev[j]) cudaEventDestroy(e->join_ev[j]);
    if (e->aux[j]) cudaStreamDestroy(e->aux[j]);
  }
  delete e;
}

}  // namespace
}  // namespace dlo

extern "C" {

dlo_status dlo_engine_create(const dlo_engine_desc* d, dlo_engine** out) {
  using namespace dlo;
  if (!d || !out) DLO_FAIL(DLO_ERR_INVALID, "dlo_engine_create: null argument");
  if (d->n_blocks < 1) DLO_FAIL(DLO_ERR_INVALID, "dlo_engine_create: n_blocks must be >= 1");
  if (!d->slot[0] || !d->slot[1] || d->slot[0] == d->slot[1])
    DLO_FAIL(DLO_ERR_INVALID, "dlo_engine_create: two distinct slots are required");
  if ((reinterpret_cast<uintptr_t>(d->slot[0]) | reinterpret_cast<uintptr_t>(d->slot[1])) & 255u)
    DLO_FAIL(DLO_ERR_INVALID, "dlo_engine_create: slots must be 256-byte aligned");
  if (d->slot_bytes <= 0) DLO_FAIL(DLO_ERR_INVALID, "dlo_engine_create: slot_bytes must be > 0");
  if (d->compute_stream == d->copy_stream)
    DLO_FAIL(DLO_ERR_INVALID, "dlo_engine_create: compute and copy streams must differ");
  if (d->copy_mode < DLO_COPY_AUTO || d->copy_mode > DLO_COPY_STAGED)
    DLO_FAIL(DLO_ERR_INVALID, "dlo_engine_create: unknown copy mode %d", d->copy_mode);
  if (d->copy_mode == DLO_COPY_STAGED) {
    if (!d->staging[0] || !d->staging[1] || d->staging[0] == d->staging[1] ||
        d->staging_bytes <= 0)
      DLO_FAIL(DLO_ERR_INVALID, "dlo_engine_create: staged copies need two staging buffers");
    if ((reinterpret_cast<uintptr_t>(d->staging[0]) |
         reinterpret_cast<uintptr_t>(d->staging[1])) & 255u)
      DLO_FAIL(DLO_ERR_INVALID, "dlo_engine_create: staging buffers must be 256-byte aligned");
    if (!d->gather_stream || d->gather_stream == d->copy_stream ||
        d->gather_stream == d->compute_stream)
      DLO_FAIL(DLO_ERR_INVALID,
               "dlo_engine_create: staged copies need a gather stream of their own");
  }
  if (d->host_staging[0] || d->host_staging[1]) {
    if (!d->host_staging[0] || !d->host_staging[1] || d->host_staging[0] == d->host_staging[1] ||
        d->host_staging_bytes <= 0)
      DLO_FAIL(DLO_ERR_INVALID, "dlo_engine_create: host staging needs two distinct buffers");
    if (d->pack_threads < 0 || d->pack_threads > 64)
      DLO_FAIL(DLO_ERR_INVALID, "dlo_engine_create: pack_threads must be 0..64");
  }
  if (d->log_capacity < 0 || d->log_capacity > (1 << 24))
    DLO_FAIL(DLO_ERR_INVALID, "dlo_engine_create: log_capacity must be 0..%d", 1 << 24);
  if (d->dma_streams < 0 || d->dma_streams > dlo_engine::kMaxFan)
    DLO_FAIL(DLO_ERR_INVALID, "dlo_engine_create: dma_streams must be 0..%d",
             dlo_engine::kMaxFan);
  DLO_TRY(preload_kernels());
  for (int s = 0; s < 2 && d->host_staging[0]; ++s) {
    cudaPointerAttributes pa{};
    const uint8_t* hs = static_cast<const uint8_t*>(d->host_staging[s]);
    if (cudaPointerGetAttributes(&pa, hs) != cudaSuccess || pa.type != cudaMemoryTypeHost ||
        cudaPointerGetAttributes(&pa, hs + d->host_staging_bytes - 1) != cudaSuccess ||
        pa.type != cudaMemoryTypeHost) {
      cudaGetLastError();
      DLO_FAIL(DLO_ERR_INVALID, "dlo_engine_create: host staging %d is not page-locked", s);
    }
  }
  dlo_engine* e = new (std::nothrow) dlo_engine();
  if (!e) DLO_FAIL(DLO_ERR_INVALID, "dlo_engine_create: out of host memory");
  e->n_blocks = d->n_blocks;
  e->slot[0] = static_cast<uint8_t*>(d->slot[0]);
  e->slot[1] = static_cast<uint8_t*>(d->slot[1]);
  e->slot_bytes = d->slot_bytes;
  e->compute = static_cast<cudaStream_t>(d->compute_stream);
  e->copy = static_cast<cudaStream_t>(d->copy_stream);
  e->slot_copy[0] = e->slot_copy[1] = e->copy;
  e->mode = d->copy_mode;
  e->copy_ctas = d->copy_ctas;
  e->timing = d->timing != 0;
  e->poison = d->poison != 0;
  e->checks = d->checks != 0;
  e->fan = d->dma_streams == 0 ? 1 : d->dma_streams;
  const size_t log_cap = d->log_capacity > 0 ? static_cast<size_t>(d->log_capacity)
                                             : static_cast<size_t>(kDefaultLogCapacity);
  e->log.set_capacity(log_cap);
  e->timed.set_capacity(log_cap);
  if (d->copy_mode == DLO_COPY_STAGED) {
    e->staging[0] = static_cast<uint8_t*>(d->staging[0]);
    e->staging[1] = static_cast<uint8_t*>(d->staging[1]);
    e->staging_bytes = d->staging_bytes;
    e->gather = static_cast<cudaStream_t>(d->gather_stream);
  }
  e->blocks.resize(d->n_blocks);
  e->hooks.resize(d->n_blocks);
  for (int32_t i = 0; i < d->n_blocks; ++i) e->hooks[i] = {i % 2, -1};
  if (d->copy_mode != DLO_COPY_AUTO) e->chosen = d->copy_mode;
  bool ok = true;
  for (int s = 0; s < 2; ++s)
    ok = ok && cudaEventCreateWithFlags(&e->ready[s], cudaEventDisableTiming) == cudaSuccess &&
         cudaEventCreateWithFlags(&e->freed[s], cudaEventDisableTiming) == cudaSuccess;
  for (int i = 0; i < 2 * kRaceWindows; ++i)
    ok = ok && cudaEventCreate(&e->race_ev[i]) == cudaSuccess;
  if (d->host_staging[0]) {
    e->host_staging[0] = static_cast<uint8_t*>(d->host_staging[0]);
    e->host_staging[1] = static_cast<uint8_t*>(d->host_staging[1]);
    e->host_staging_bytes = d->host_staging_bytes;
    for (int s = 0; s < 2; ++s)
      ok = ok && cudaEventCreateWithFlags(&e->hs_read[s], cudaEventDisableTiming) == cudaSuccess;
  }
  if (d->two_copy_streams) {
    ok = ok && cudaStreamCreateWithFlags(&e->own_copy, cudaStreamNonBlocking) == cudaSuccess;
    e->slot_copy[1] = e->own_copy;
  }
  e->pool = new (std::nothrow) PackPool(d->pack_threads > 0 ? d->pack_threads : 4);
  ok = ok && e->pool != nullptr;
  if (e->gather)
    for (int s = 0; s < 2; ++s)
      ok = ok &&
           cudaEventCreateWithFlags(&e->staged[s], cudaEventDisableTiming) == cudaSuccess &&
           cudaEventCreateWithFlags(&e->stage_free[s], cudaEventDisableTiming) == cudaSuccess;
  ok = ok && cudaStreamCreateWithFlags(&e->side, cudaStreamNonBlocking) == cudaSuccess &&
       cudaEventCreateWithFlags(&e->side_fork, cudaEventDisableTiming) == cudaSuccess &&
       cudaEventCreateWithFlags(&e->side_join, cudaEventDisableTiming) == cudaSuccess;
  if (e->fan > 1) {
    ok = ok && cudaEventCreateWithFlags(&e->fork_ev, cudaEventDisableTiming) == cudaSuccess;
    for (int j = 0; j < e->fan; ++j)
      ok = ok && cudaStreamCreateWithFlags(&e->aux[j], cudaStreamNonBlocking) == cudaSuccess &&
           cudaEventCreateWithFlags(&e->join_ev[j], cudaEventDisableTiming) == cudaSuccess;
  }
  if (!ok) {
    cudaGetLastError();
    release(e);
    DLO_FAIL(DLO_ERR_CUDA, "dlo_engine_create: cannot create the engine's events/streams");
  }
  *out = e;
  return DLO_OK;
}

}  // extern "C"

namespace dlo {
namespace {

// A block's shard table from the caller's pointers: each shard non-null,
// 16-byte aligned and page-locked host memory (its device-mapped address
// kept for the copy kernel).
dlo_status shard_table(const char* who, const dlo_plan* plan, const void* const* shard_ptrs,
                       dlo_engine::Block* b) {
  const size_t n = plan->groups.size() * static_cast<size_t>(plan->n_shards);
  if (n > static_cast<size_t>(kMaxSegments))
    DLO_FAIL(DLO_ERR_INVALID, "%s: %zu (group, shard) pieces, at most %d", who, n,
             kMaxSegments);
  b->plan = plan;
  b->host.assign(shard_ptrs, shard_ptrs + n);
  b->dev.assign(n, nullptr);
  b->bytes = 0;
  for (size_t i = 0; i < n; ++i) {
    const void* q = shard_ptrs[i];
    if (!q || (reinterpret_cast<uintptr_t>(q) & 15u))
      DLO_FAIL(DLO_ERR_INVALID, "%s: shard %zu is null or not 16-byte aligned", who, i);
    cudaPointerAttributes a{};
    if (cudaPointerGetAttributes(&a, q) != cudaSuccess || a.type != cudaMemoryTypeHost) {
      cudaGetLastError();
      DLO_FAIL(DLO_ERR_INVALID, "%s: shard %zu is not page-locked host memory", who, i);
    }
    b->dev[i] = a.devicePointer;
  }
  for (const auto& g : plan->groups) b->bytes += g.shard_bytes * plan->n_shards;
  compute_pitches(b);
  return DLO_OK;
}

}  // namespace
}  // namespace dlo

extern "C" {

dlo_status dlo_register_block(dlo_engine* e, int32_t block, const dlo_plan* plan,
                              const void* const* shard_ptrs) {
  using namespace dlo;
  DLO_TRY(check_engine(e));
  if (block < 0 || block >= e->n_blocks)
    DLO_FAIL(DLO_ERR_INVALID, "dlo_register_block: block %d out of range", block);
  if (!plan || !shard_ptrs) DLO_FAIL(DLO_ERR_INVALID, "dlo_register_block: null argument");
  if (e->blocks[block].plan)
    DLO_FAIL(DLO_ERR_STATE, "dlo_register_block: block %d already registered", block);
  if (plan->slot_bytes > e->slot_bytes)
    DLO_FAIL(DLO_ERR_INVALID, "dlo_register_block: block needs %lld bytes, slots hold %lld",
             (long long)plan->slot_bytes, (long long)e->slot_bytes);
  if (e->gather && plan->staging_bytes > e->staging_bytes)
    DLO_FAIL(DLO_ERR_INVALID,
             "dlo_register_block: block needs %lld staging bytes, staging holds %lld",
             (long long)plan->staging_bytes, (long long)e->staging_bytes);
  dlo_engine::Block b;
  DLO_TRY(shard_table("dlo_register_block", plan, shard_ptrs, &b));
  if (e->mode == DLO_COPY_KERNEL && !all_mapped(b))
    DLO_FAIL(DLO_ERR_INVALID, "dlo_register_block: kernel copies need device-mapped shards");
  e->blocks[block] = std::move(b);
  return DLO_OK;
}

dlo_status dlo_replace_block_shards(dlo_engine* e, int32_t block,
                                    const void* const* shard_ptrs, int32_t timeout_ms) {
  using namespace dlo;
  DLO_TRY(check_engine(e));
  if (block < 0 || block >= e->n_blocks || !shard_ptrs)
    DLO_FAIL(DLO_ERR_INVALID, "dlo_replace_block_shards: bad block %d or null pointers", block);
  const dlo_engine::Block& cur = e->blocks[block];
  if (!cur.plan || cur.source)
    DLO_FAIL(DLO_ERR_STATE, "dlo_replace_block_shards: block %d has no registered shards",
             block);
  TraceRange range("replace_block_shards", block);
  dlo_engine::Block b;
  DLO_TRY(shard_table("dlo_replace_block_shards", cur.plan, shard_ptrs, &b));
  if (e->mode == DLO_COPY_KERNEL && !all_mapped(b))
    DLO_FAIL(DLO_ERR_INVALID,
             "dlo_replace_block_shards: kernel copies need device-mapped shards");
  // every copy already enqueued from the old shards (a slot holding the
  // block has one pending until its ready event completes) must finish
  // before the caller may reuse that memory
  for (int s = 0; s < 2; ++s)
    if (e->slot_holds[s] == block && !wait_event_host(e->ready[s], timeout_ms))
      DLO_FAIL(DLO_ERR_TIMEOUT,
               "dlo_replace_block_shards: block %d's copy into slot %d not done after %d ms",
               block, s, timeout_ms);
  e->blocks[block] = std::move(b);
  return DLO_OK;
}

dlo_status dlo_register_block_source(dlo_engine* e, int32_t block, const dlo_plan* plan,
                                     const void* const* param_src) {
  using namespace dlo;
  DLO_TRY(check_engine(e));
  if (block < 0 || block >= e->n_blocks)
    DLO_FAIL(DLO_ERR_INVALID, "dlo_register_block_source: block %d out of range", block);
  if (!plan || !param_src) DLO_FAIL(DLO_ERR_INVALID, "dlo_register_block_source: null argument");
  if (e->blocks[block].plan)
    DLO_FAIL(DLO_ERR_STATE, "dlo_register_block_source: block %d already registered", block);
  if (plan->n_shards != 1)
    DLO_FAIL(DLO_ERR_INVALID, "dlo_register_block_source: the rank-local path has 1 shard");
  if (plan->slot_bytes > e->slot_bytes)
    DLO_FAIL(DLO_ERR_INVALID, "dlo_register_block_source: block needs %lld bytes, slots hold %lld",
             (long long)plan->slot_bytes, (long long)e->slot_bytes);
  dlo_engine::Block b;
  b.plan = plan;
  b.source = true;
  b.direct = true;
  for (size_t p = 0; p < plan->params.size(); ++p) {
    const auto& q = plan->params[p];
    const uint8_t* s = static_cast<const uint8_t*>(param_src[p]);
    if (!s) DLO_FAIL(DLO_ERR_INVALID, "dlo_register_block_source: param %zu is null", p);
    const int64_t n = q.storage_numel * plan->groups[q.group].esize;
    b.src.push_back({s, n, q.slot_offset});
    b.bytes += n;
    cudaPointerAttributes a0{}, a1{};
    const bool locked = cudaPointerGetAttributes(&a0, s) == cudaSuccess &&
                        a0.type == cudaMemoryTypeHost &&
                        cudaPointerGetAttributes(&a1, s + n - 1) == cudaSuccess &&
                        a1.type == cudaMemoryTypeHost;
    cudaGetLastError();
    b.direct = b.direct && locked;
  }
  if (!b.direct && (!e->host_staging[0] || e->host_staging_bytes < plan->slot_bytes))
    DLO_FAIL(DLO_ERR_INVALID,
             "dlo_register_block_source: pageable parameters need host staging of %lld bytes",
             (long long)plan->slot_bytes);
  e->blocks[block] = std::move(b);
  return DLO_OK;
}

dlo_status dlo_prefetch(dlo_engine* e, int32_t block, int32_t slot) {
  using namespace dlo;
  DLO_TRY(check_engine(e));
  if (block < 0 || block >= e->n_blocks || slot < 0 || slot > 1)
    DLO_FAIL(DLO_ERR_INVALID, "dlo_prefetch: block %d / slot %d out of range", block, slot);
  if (!e->blocks[block].plan)
    DLO_FAIL(DLO_ERR_STATE, "dlo_prefetch: block %d is not registered", block);
  if (e->in_forward && e->cur_slot == slot)
    DLO_FAIL(DLO_ERR_STATE, "dlo_prefetch: slot %d is being read by block %d", slot,
             e->cur_block);
  return enqueue_prefetch(e, block, slot, -1);
}

dlo_status dlo_wait(dlo_engine* e, int32_t block) {
  using namespace dlo;
  DLO_TRY(check_engine(e));
  const int32_t s = slot_of(e, block);
  if (s < 0) DLO_FAIL(DLO_ERR_STATE, "dlo_wait: block %d is in no slot", block);
  DLO_CUDA(cudaStreamWaitEvent(e->compute, e->ready[s], 0));
  return DLO_OK;
}

dlo_status dlo_wait_host(dlo_engine* e, int32_t block, int32_t timeout_ms) {
  using namespace dlo;
  DLO_TRY(check_engine(e));
  TraceRange range("wait_host", block);
  const int32_t s = slot_of(e, block);
  if (s < 0) DLO_FAIL(DLO_ERR_STATE, "dlo_wait_host: block %d is in no slot", block);
  const auto t0 = std::chrono::steady_clock::now();
  for (;;) {
    const cudaError_t q = cudaEventQuery(e->ready[s]);
    if (q == cudaSuccess) return DLO_OK;
    if (q != cudaErrorNotReady) DLO_CUDA(q);
    const auto ms = std::chrono::duration_cast<std::chrono::milliseconds>(
                        std::chrono::steady_clock::now() - t0)
                        .count();
    if (ms >= timeout_ms)
      DLO_FAIL(DLO_ERR_TIMEOUT, "dlo_wait_host: block %d not ready after %d ms", block,
               timeout_ms);
    std::this_thread::sleep_for(std::chrono::microseconds(50));
  }
}

dlo_status dlo_param_view(const dlo_engine* e, int32_t block, int32_t param, void** dev_ptr) {
  using namespace dlo;
  DLO_TRY(check_engine(e));
  if (!dev_ptr) DLO_FAIL(DLO_ERR_INVALID, "dlo_param_view: null argument");
  if (block < 0 || block >= e->n_blocks || !e->blocks[block].plan)
    DLO_FAIL(DLO_ERR_INVALID, "dlo_param_view: block %d not registered", block);
  const dlo_plan* p = e->blocks[block].plan;
  if (param < 0 || param >= static_cast<int32_t>(p->params.size()))
    DLO_FAIL(DLO_ERR_INVALID, "dlo_param_view: param %d out of range", param);
  const int32_t s = slot_of(e, block);
  if (s < 0) DLO_FAIL(DLO_ERR_STATE, "dlo_param_view: block %d is in no slot", block);
  if (e->checks) {
    // the view's bytes: its elements' place in the flat group, which lies
    // inside the group's gathered elements and the slot
    const auto& q = p->params[param];
    const auto& grp = p->groups[q.group];
    const int64_t lo = q.slot_offset, hi = lo + q.storage_numel * grp.esize;
    if (lo != grp.base + q.group_offset * grp.esize || q.group_offset < 0 ||
        q.group_offset + q.storage_numel > grp.numel || hi > e->slot_bytes)
      DLO_FAIL(DLO_ERR_STATE, "dlo_param_view: param %d's bytes [%lld, %lld) are not its "
               "elements [%lld, %lld) of group %d at base %lld", param, (long long)lo,
               (long long)hi, (long long)q.group_offset,
               (long long)(q.group_offset + q.storage_numel), q.group, (long long)grp.base);
  }
  *dev_ptr = e->slot[s] + p->params[param].slot_offset;
  return DLO_OK;
}

dlo_status dlo_pre_forward(dlo_engine* e, int32_t block, int32_t* slot_out) {
  using namespace dlo;
  DLO_TRY(check_engine(e));
  TraceRange range("pre_forward", block);
  if (e->in_forward)
    DLO_FAIL(DLO_ERR_STATE, "dlo_pre_forward: block %d has no post_forward yet", e->cur_block);
  const int32_t n = e->n_blocks;
  const int32_t expect = static_cast<int32_t>(e->k % n);
  if (block != expect)
    DLO_FAIL(DLO_ERR_STATE, "dlo_pre_forward: forward %lld must run block %d, not %d",
             (long long)e->k, expect, block);
  const int32_t next = (block + 1) % n;
  if (!e->blocks[block].plan || !e->blocks[next].plan)
    DLO_FAIL(DLO_ERR_STATE, "dlo_pre_forward: block %d or %d is not registered", block, next);
  dlo_engine::Hook& h = e->hooks[block];
  const dlo_engine::Hook& prev = e->hooks[(block + n - 1) % n];
  int32_t slot = h.current_slot;
  if (prev.prefetched_slot >= 0) slot = prev.prefetched_slot;
  if (e->slot_holds[slot] != block)
    DLO_FAIL(DLO_ERR_STATE, "dlo_pre_forward: slot %d holds block %d, not %d", slot,
             e->slot_holds[slot], block);
  DLO_CUDA(cudaStreamWaitEvent(e->compute, e->ready[slot], 0));
  const int32_t ps = 1 - slot;
  const int32_t waits = e->last_reader[ps];
  int32_t used_mode = DLO_COPY_DMA;
  DLO_TRY(enqueue_prefetch(e, next, ps, e->k, &used_mode));
  h.current_slot = slot;
  h.prefetched_slot = ps;
  e->last_reader[slot] = static_cast<int32_t>(e->k);
  dlo_sched_event ev;
  ev.k = static_cast<int32_t>(e->k);
  ev.block = block;
  ev.read_slot = slot;
  ev.prefetch_block = next;
  ev.prefetch_slot = ps;
  ev.waits_on_free_of_k = waits;
  ev.copy_mode = used_mode;
  bool reused = false;
  e->log.push(&reused) = ev;
  e->in_forward = true;
  e->cur_block = block;
  e->cur_slot = slot;
  if (slot_out) *slot_out = slot;
  return DLO_OK;
}

dlo_status dlo_post_forward(dlo_engine* e, int32_t block) {
  using namespace dlo;
  DLO_TRY(check_engine(e));
  TraceRange range("post_forward", block);
  if (!e->in_forward || block != e->cur_block)
    DLO_FAIL(DLO_ERR_STATE, "dlo_post_forward: block %d is not the block in flight", block);
  if (e->poison)
    DLO_CUDA(cudaMemsetAsync(e->slot[e->cur_slot], 0xA5, static_cast<size_t>(e->slot_bytes),
                             e->compute));
  DLO_CUDA(cudaEventRecord(e->freed[e->cur_slot], e->compute));
  if (e->chosen < 0) {
    const int64_t s0 = race_start(e->n_blocks);
    for (int w = 0; w < kRaceWindows; ++w) {
      const int64_t first = s0 + w * kRaceWindow, lastk = first + kRaceWindow - 1;
      if (e->k == first || e->k == lastk) {
        const int i = 2 * w + (e->k == lastk ? 1 : 0);
        DLO_CUDA(cudaEventRecord(e->race_ev[i], e->compute));
        e->race_rec[i] = true;
      }
    }
  }
  e->in_forward = false;
  e->k++;
  return DLO_OK;
}

dlo_status dlo_block_forward(dlo_engine* e, int32_t block, const dlo_dit_cfg* cfg, float* x,
                             void* scratch, size_t scratch_bytes) {
  using namespace dlo;
  DLO_TRY(check_engine(e));
  TraceRange range("block_forward", block);
  int32_t slot = -1;
  DLO_TRY(dlo_pre_forward(e, block, &slot));
  const dlo_status st = forward_impl(cfg, e->blocks[block].plan, e->slot[slot], x, scratch,
                                     scratch_bytes, e->compute);
  // the free event is recorded even if a launch was refused, so that the
  // schedule stays consistent; the error is still returned
  const dlo_status st2 = dlo_post_forward(e, block);
  return st != DLO_OK ? st : st2;
}

dlo_status dlo_schedule_log(const dlo_engine* e, dlo_sched_event* buf, int32_t cap,
                            int32_t* n_out) {
  using namespace dlo;
  DLO_TRY(check_engine(e));
  if (!n_out || (cap > 0 && !buf)) DLO_FAIL(DLO_ERR_INVALID, "dlo_schedule_log: null argument");
  const int32_t n = static_cast<int32_t>(e->log.size());
  const int32_t m = n < cap ? n : cap;
  // the newest m entries, oldest first
  for (int32_t i = 0; i < m; ++i) buf[i] = e->log.at(static_cast<size_t>(n - m + i));
  *n_out = n;
  return DLO_OK;
}

dlo_status dlo_engine_query(dlo_engine* e, dlo_engine_stats* out) {
  using namespace dlo;
  DLO_TRY(check_engine(e));
  if (!out) DLO_FAIL(DLO_ERR_INVALID, "dlo_engine_query: null argument");
  try_decide(e);
  out->chosen_mode = e->chosen >= 0 ? e->chosen : DLO_COPY_AUTO;
  out->n_forwards = static_cast<int32_t>(e->k);
  out->n_prefetches = static_cast<int32_t>(e->n_prefetches);
  out->n_kernel_prefetches = static_cast<int32_t>(e->n_kernel_prefetches);
  out->race_dma_us = e->race_dma_us;
  out->race_kernel_us = e->race_kernel_us;
  out->n_direct_prefetches = static_cast<int32_t>(e->n_direct);
  out->n_packed_prefetches = static_cast<int32_t>(e->n_packed);
  out->pack_ms = e->pack_ms;
  out->n_copy_kernel_launches = static_cast<int32_t>(e->n_copy_launches);
  out->log_dropped = e->log.dropped();
  out->timed_dropped = e->timed.dropped();
  out->checked_pieces = e->checked_pieces;
  return DLO_OK;
}

dlo_status dlo_engine_copy_times(dlo_engine* e, float* copy_ms, int64_t* copy_bytes, int32_t cap,
                                 int32_t* n_out) {
  using namespace dlo;
  DLO_TRY(check_engine(e));
  if (!n_out || (cap > 0 && (!copy_ms || !copy_bytes)))
    DLO_FAIL(DLO_ERR_INVALID, "dlo_engine_copy_times: null argument");
  const int32_t n = static_cast<int32_t>(e->timed.size());
  for (int32_t i = 0; i < n && i < cap; ++i) {
    const dlo_engine::Timed& t = e->timed.at(static_cast<size_t>(i));
    DLO_CUDA(cudaEventSynchronize(t.b));
    float ms = 0;
    DLO_CUDA(cudaEventElapsedTime(&ms, t.a, t.b));
    copy_ms[i] = ms;
    copy_bytes[i] = t.bytes;
  }
  *n_out = n;
  return DLO_OK;
}

dlo_status dlo_engine_copy_spans(dlo_engine* e, float* start_ms, float* end_ms, int32_t cap,
                                 int32_t* n_out) {
  using namespace dlo;
  DLO_TRY(check_engine(e));
  if (!n_out || (cap > 0 && (!start_ms || !end_ms)))
    DLO_FAIL(DLO_ERR_INVALID, "dlo_engine_copy_spans: null argument");
  const int32_t n = static_cast<int32_t>(e->timed.size());
  for (int32_t i = 0; i < n && i < cap; ++i) {
    const dlo_engine::Timed& t = e->timed.at(static_cast<size_t>(i));
    const cudaEvent_t origin = e->timed.at(0).a;
    DLO_CUDA(cudaEventSynchronize(t.b));
    float a = 0, b = 0;
    DLO_CUDA(cudaEventElapsedTime(&a, origin, t.a));
    DLO_CUDA(cudaEventElapsedTime(&b, origin, t.b));
    start_ms[i] = a;
    end_ms[i] = b;
  }
  *n_out = n;
  return DLO_OK;
}

dlo_status dlo_engine_copy_log(dlo_engine* e, int64_t since, dlo_copy_record* buf, int32_t cap,
                               int32_t* n_out, int64_t* next) {
  using namespace dlo;
  DLO_TRY(check_engine(e));
  if (!n_out || !next || (cap > 0 && !buf))
    DLO_FAIL(DLO_ERR_INVALID, "dlo_engine_copy_log: null argument");
  const size_t kept = e->timed.size();
  int64_t seq = since;
  if (kept > 0 && seq < e->timed.at(0).seq) seq = e->timed.at(0).seq;   // older ones dropped
  int32_t n = 0;
  if (kept > 0) {
    for (size_t i = static_cast<size_t>(seq - e->timed.at(0).seq); i < kept && n < cap; ++i) {
      const dlo_engine::Timed& t = e->timed.at(i);
      const cudaError_t q = cudaEventQuery(t.b);
      if (q == cudaErrorNotReady) break;        // not done yet: report it next time
      DLO_CUDA(q);
      float ms = 0;
      DLO_CUDA(cudaEventElapsedTime(&ms, t.a, t.b));
      buf[n].seq = t.seq;
      buf[n].block = t.block;
      buf[n].slot = t.slot;
      buf[n].copy_ms = ms;
      buf[n].bytes = t.bytes;
      ++n;
      seq = t.seq + 1;
    }
  }
  *n_out = n;
  *next = seq;
  return DLO_OK;
}

dlo_status dlo_engine_destroy(dlo_engine* e, int32_t timeout_ms) {
  using namespace dlo;
  if (!e) return DLO_OK;
  TraceRange range("engine_destroy", e->n_blocks);
  // drain the streams (bounded): mark their current tails and poll
  cudaEvent_t tail[4] = {nullptr, nullptr, nullptr, nullptr};
  cudaStream_t st[4] = {e->copy, e->compute, nullptr, nullptr};
  int n = 2;
  if (e->own_copy) st[n++] = e->own_copy;
  if (e->gather) st[n++] = e->gather;
  auto drop = [&]() {
    for (int i = 0; i < n; ++i)
      if (tail[i]) cudaEventDestroy(tail[i]);
  };
  for (int i = 0; i < n; ++i) {
    if (cudaEventCreateWithFlags(&tail[i], cudaEventDisableTiming) != cudaSuccess ||
        cudaEventRecord(tail[i], st[i]) != cudaSuccess) {
      drop();
      DLO_FAIL(DLO_ERR_CUDA, "dlo_engine_destroy: cannot mark the stream tails");
    }
  }
  const auto t0 = std::chrono::steady_clock::now();
  for (;;) {
    bool done = true;
    for (int i = 0; i < n; ++i) {
      const cudaError_t q = cudaEventQuery(tail[i]);
      if (q == cudaErrorNotReady) {
        done = false;
      } else if (q != cudaSuccess) {
        drop();
        DLO_FAIL(DLO_ERR_CUDA, "dlo_engine_destroy: stream error while draining");
      }
    }
    if (done) break;
    const auto ms = std::chrono::duration_cast<std::chrono::milliseconds>(
                        std::chrono::steady_clock::now() - t0)
                        .count();
    if (ms >= timeout_ms) {
      drop();
      DLO_FAIL(DLO_ERR_TIMEOUT, "dlo_engine_destroy: streams not drained after %d ms",
               timeout_ms);
    }
    std::this_thread::sleep_for(std::chrono::microseconds(100));
  }
  drop();
  release(e);
  return DLO_OK;
}

dlo_status dlo_reassemble(const dlo_plan* plan, const void* const* shard_ptrs, void* dst,
                          int32_t mode, void* stream) {
  using namespace dlo;
  if (!plan || !shard_ptrs || !dst) DLO_FAIL(DLO_ERR_INVALID, "dlo_reassemble: null argument");
  TraceRange range("reassemble", plan->slot_bytes);
  if (reinterpret_cast<uintptr_t>(dst) & 255u)
    DLO_FAIL(DLO_ERR_INVALID, "dlo_reassemble: dst must be 256-byte aligned");
  const size_t n = plan->groups.size() * static_cast<size_t>(plan->n_shards);
  if (n > static_cast<size_t>(kMaxSegments))
    DLO_FAIL(DLO_ERR_INVALID, "dlo_reassemble: too many (group, shard) pieces");
  dlo_engine::Block b;
  b.plan = plan;
  b.host.assign(shard_ptrs, shard_ptrs + n);
  b.dev.assign(n, nullptr);
  for (size_t i = 0; i < n; ++i) {
    const void* q = shard_ptrs[i];
    if (!q || (reinterpret_cast<uintptr_t>(q) & 15u))
      DLO_FAIL(DLO_ERR_INVALID, "dlo_reassemble: shard %zu null or not 16-byte aligned", i);
    if (mode == DLO_COPY_KERNEL) {
      cudaPointerAttributes a{};
      if (cudaPointerGetAttributes(&a, q) != cudaSuccess || a.type != cudaMemoryTypeHost ||
          !a.devicePointer) {
        cudaGetLastError();
        DLO_FAIL(DLO_ERR_INVALID, "dlo_reassemble: shard %zu is not mapped pinned memory", i);
      }
      b.dev[i] = a.devicePointer;
    }
  }
  if (mode == DLO_COPY_STAGED)
    DLO_FAIL(DLO_ERR_INVALID, "dlo_reassemble: staged copies go through dlo_reassemble_staged");
  const int32_t m = mode == DLO_COPY_KERNEL ? DLO_COPY_KERNEL : DLO_COPY_DMA;
  compute_pitches(&b);
  return copy_block(b, static_cast<uint8_t*>(dst), m, 0, static_cast<cudaStream_t>(stream), 1,
                    nullptr, nullptr, nullptr);
}

dlo_status dlo_reassemble_staged(const dlo_plan* plan, const void* const* shard_ptrs,
                                 void* staging, int64_t staging_bytes, void* dst,
                                 void* copy_stream, void* gather_stream) {
  using namespace dlo;
  if (!plan || !shard_ptrs || !staging || !dst)
    DLO_FAIL(DLO_ERR_INVALID, "dlo_reassemble_staged: null argument");
  TraceRange range("reassemble_staged", plan->slot_bytes);
  if ((reinterpret_cast<uintptr_t>(dst) | reinterpret_cast<uintptr_t>(staging)) & 255u)
    DLO_FAIL(DLO_ERR_INVALID, "dlo_reassemble_staged: dst and staging must be 256-byte aligned");
  if (staging_bytes < plan->staging_bytes)
    DLO_FAIL(DLO_ERR_INVALID, "dlo_reassemble_staged: staging holds %lld bytes, needs %lld",
             (long long)staging_bytes, (long long)plan->staging_bytes);
  const size_t n = plan->groups.size() * static_cast<size_t>(plan->n_shards);
  if (n > static_cast<size_t>(kMaxSegments))
    DLO_FAIL(DLO_ERR_INVALID, "dlo_reassemble_staged: too many (group, shard) pieces");
  dlo_engine::Block b;
  b.plan = plan;
  b.host.assign(shard_ptrs, shard_ptrs + n);
  for (size_t i = 0; i < n; ++i)
    if (!shard_ptrs[i] || (reinterpret_cast<uintptr_t>(shard_ptrs[i]) & 15u))
      DLO_FAIL(DLO_ERR_INVALID, "dlo_reassemble_staged: shard %zu null or not 16-byte aligned",
               i);
  compute_pitches(&b);
  const cudaStream_t cs = static_cast<cudaStream_t>(copy_stream);
  const cudaStream_t gs = static_cast<cudaStream_t>(gather_stream);
  DLO_TRY(stage_h2d(b, static_cast<uint8_t*>(staging), cs));
  if (gs != cs) {
    cudaEvent_t ev = nullptr;
    DLO_CUDA(cudaEventCreateWithFlags(&ev, cudaEventDisableTiming));
    const cudaError_t e1 = cudaEventRecord(ev, cs);
    const cudaError_t e2 = e1 == cudaSuccess ? cudaStreamWaitEvent(gs, ev, 0) : e1;
    cudaEventDestroy(ev);   // released once the recorded work completes
    DLO_CUDA(e2);
  }
  return stage_gather(plan, static_cast<const uint8_t*>(staging), static_cast<uint8_t*>(dst), 0,
                      gs);
}

}  // extern "C"
