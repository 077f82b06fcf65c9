/*
 * dlo.h — C ABI of the GB300 per-block weight stream of Distributed
 * Layerwise Offload (DLO).
 *
 * Sources, cited by page title and section:
 *   [B1] "Distributed Layerwise Offload" (vLLM blog preview, 2026-07-30):
 *        "Weight Sharding + AllGather", "Double-Buffer Memory Bound",
 *        "Slot Tracking: i%2 + Dynamic Correction", "Fail-Closed Design".
 *   [B2] "Distributed Layerwise Offload: Scaling Toward 200B+ DiT Models
 *        Efficiently in vLLM-Omni" (vLLM blog, 2026-08-17):
 *        "2. Weight Sharding with AllGather Reconstruction",
 *        "3. Double-Buffered Prefetch with H2D + AllGather Overlap".
 *   [D5] vLLM-Omni design doc "Distributed Layerwise Offload":
 *        "AllGather path", "Rank-local path without DLO AllGather".
 *
 * What the library does.  Each block's parameters are flattened by dtype and
 * split into n_shards equal, zero-padded shards that live in pinned host
 * memory.  Two device slots, each large enough for the largest block, hold
 * the block being computed and the block being prefetched.  A prefetch copies
 * every shard host->device and reassembles the shards, in rank order, into
 * the slot (on one GPU the n_shards host regions stand in for the ranks of an
 * all_gather_into_tensor).  Parameters are zero-copy pointers into the slot.
 * The block forward runs on a compute stream that waits for the slot's ready
 * event; the next block's prefetch runs on a copy stream that waits for the
 * free event of the forward that last read the target slot.
 *
 * Conventions.
 *   - Every call returns a dlo_status.  Out-parameters are written only on
 *     DLO_OK.  On failure dlo_last_error() returns a message (per thread).
 *     Nothing throws across the ABI.  Calls fail closed ([B1] "Fail-Closed
 *     Design"): a call that would read a slot that does not hold the
 *     requested block, or write a slot that is still being read without a
 *     wait, returns an error instead.
 *   - Streams are passed as `void*` holding a cudaStream_t; device and host
 *     buffers as plain pointers.  The header needs no CUDA include.
 *   - bf16 tensors are passed as uint16_t (raw bits).
 *   - The library never allocates device memory or pins host memory: the
 *     caller owns slots, activations, scratch, shard buffers and streams.
 *     The library owns plans, engines, their CUDA events and logs.
 *   - Tracing: the plan, shard, hook, prefetch, forward, reassembly and
 *     teardown calls push NVTX ranges in the domain "dlo" (payload: the
 *     block index for hooks and prefetches, the number of rows for a
 *     forward, the number of parameters for plan_create and shard_host, the
 *     slot bytes for a one-shot reassembly).  Without an NVTX tool attached
 *     (nsys, ncu --nvtx, or a library named by NVTX_INJECTION64_PATH) they
 *     cost a load and a branch each.
 */
#ifndef DLO_H_
#define DLO_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  DLO_OK = 0,
  DLO_ERR_INVALID = 1,  /* bad argument: null, size, alignment, unknown name */
  DLO_ERR_CUDA = 2,     /* a CUDA runtime/driver call failed (text in dlo_last_error) */
  DLO_ERR_TIMEOUT = 3,  /* a bounded wait ran out (host poll or device-side wait) */
  DLO_ERR_STATE = 4,    /* call not valid in the current state (e.g. block not resident) */
  DLO_ERR_NOMEM = 5,    /* a caller-provided buffer is too small */
  DLO_ERR_PARTIAL = 6   /* a registration failed and could not be fully rolled
                           back: some ranges are still registered, so their
                           mappings must stay open (fatal for the caller's
                           setup) */
} dlo_status;

/* Element types of parameters.  Every distinct code forms its own dtype
 * group (its own flat buffer and shards), so an 8-bit weight and its 8-bit
 * block scales travel as two groups.  The 1-byte codes cover the layouts the
 * pages' online quantisation keeps ("Request and loading constraints": an
 * int8 weight with an fp32 scale, an fp8 weight with an e8m0 block scale);
 * the library moves their bytes and interprets none of them. */
typedef enum {
  DLO_BF16 = 0,
  DLO_F32 = 1,
  DLO_F16 = 2,
  DLO_FP8_E4M3 = 3,
  DLO_FP8_E5M2 = 4,
  DLO_I8 = 5,
  DLO_U8 = 6,
  DLO_E8M0 = 7   /* 8-bit power-of-two block scale */
} dlo_dtype;

/* How a prefetch moves the shards host->device.
 *   DMA:    copy engines, no SMs: per dtype group one cudaMemcpy2DAsync
 *           when the group's host shards sit at a constant stride (rows =
 *           shards, destination pitch = shard bytes, i.e. the gathered
 *           layout; one cudaMemcpyAsync when that stride equals the shard
 *           bytes), else one cudaMemcpyAsync per shard, each straight to
 *           the shard's final offset in the slot.  In the engine, a group
 *           under 1 MiB (when the block has another, larger group and its
 *           shards are device-mapped) moves by a one-CTA copy-kernel launch
 *           on a library-owned side stream while the DMA runs.
 *   KERNEL: one launch of a copy-and-reassemble kernel that reads the mapped
 *           pinned host shards with 16-byte loads and writes them to their
 *           final slot offsets (SMs read over the host link).
 *   AUTO:   the first prefetches alternate between the two under the real
 *           workload, timed with events; the faster per byte is then kept.
 *   STAGED: the two-phase form of [B1] "Weight Sharding + AllGather" steps
 *           1-2 ([B2] §3: H2D on copy_stream, AllGather on comm_stream): the
 *           shards first land, by DMA, in a device staging buffer laid out
 *           shard by shard (group g, shard r at stage_base_g + r *
 *           shard_alloc_bytes); then a device-to-device copy-and-reassemble
 *           kernel on a second ("gather") stream writes them to their slot
 *           offsets, which is what all_gather_into_tensor produces.  Needs
 *           the engine's staging buffers and gather stream.  Never chosen by
 *           AUTO. */
typedef enum {
  DLO_COPY_AUTO = 0,
  DLO_COPY_DMA = 1,
  DLO_COPY_KERNEL = 2,
  DLO_COPY_STAGED = 3
} dlo_copy_mode;

/* ------------------------------------------------------------------------
 * Plan: the per-block layout ([B1] "Weight Sharding + AllGather"; [B2] §2).
 * ------------------------------------------------------------------------ */

typedef struct {
  const char* name;     /* parameter name, copied by dlo_plan_create */
  int32_t ndim;         /* 1..4 */
  int64_t shape[4];     /* logical extents */
  int32_t dtype;        /* dlo_dtype */
  int64_t stride[4];    /* element strides of the view over its storage, each
                           >= 0; all 0 means row-major contiguous.  A strided
                           view (e.g. a transposed finalized weight) is packed
                           in physical order: the plan moves its storage
                           extent, 1 + sum_i (shape[i]-1)*stride[i] elements
                           starting at element [0,..,0], and the device-side
                           view is the same strides over the slot copy
                           (reading of "physical-order packing", "Request and
                           loading constraints") */
} dlo_param_desc;

typedef struct dlo_plan dlo_plan;

typedef struct {
  int32_t n_params;
  int32_t n_groups;     /* distinct dtypes, in order of first appearance */
  int32_t n_shards;
  int32_t has_dit_roles;/* 1 if the names match the synthetic DiT block */
  int64_t slot_bytes;   /* bytes a slot needs for this block */
  int64_t group_align;  /* byte alignment of each group's base in a slot (256) */
  int64_t staging_bytes;/* bytes a staging buffer needs for this block in
                           DLO_COPY_STAGED (groups shard by shard, each shard
                           at a 16-byte aligned offset) */
} dlo_plan_info;

typedef struct {
  int32_t dtype;
  int32_t esize;            /* bytes per element */
  int64_t numel;            /* N_g: elements of all params of this dtype */
  int64_t shard_numel;      /* S_g = ceil(N_g / n_shards)  ([B2] §2) */
  int64_t shard_bytes;      /* S_g * esize: bytes each shard contributes */
  int64_t shard_alloc_bytes;/* shard_bytes rounded up to 16: required size of
                               every host shard buffer of this group */
  int64_t base;             /* byte offset of the gathered group in a slot */
  int64_t stage_base;       /* byte offset of the group's first shard in a
                               staging buffer (256-byte aligned); shard r at
                               stage_base + r * shard_alloc_bytes */
} dlo_group_info;

typedef struct {
  int32_t group;            /* index into the plan's groups */
  int32_t dtype;
  int64_t numel;            /* logical elements (product of the extents) */
  int64_t group_offset;     /* element offset inside the flat group */
  int64_t slot_offset;      /* byte offset inside a slot (base + offset*esize) */
  int64_t storage_numel;    /* elements packed for it (its storage extent;
                               numel for a contiguous parameter) */
  int64_t stride[4];        /* element strides of the device-side view
                               (row-major ones for a contiguous parameter) */
} dlo_param_info;

/* Builds the layout of one block.  Parameters of one dtype are concatenated
 * in the given (registration) order with no gap; each dtype group is split
 * into n_shards shards of S_g = ceil(N_g / n_shards) elements, the last
 * zero-padded ([B2] §2); in a slot, groups follow in order of first
 * appearance, each at a 256-byte aligned base, each occupying
 * n_shards * S_g elements (the gathered buffer, padding included).
 * n_shards >= 1 (1 is the rank-local path of [D5]).  *out is owned by the
 * caller and released with dlo_plan_destroy.  Parameters of different
 * blocks may differ in number, names, dtypes and sizes (heterogeneous
 * blocks): each block has its own plan, and an engine's slots must hold the
 * largest.  has_dit_roles is set when all twelve DiT parameter names are
 * present with the dtypes the block forward reads (bf16 linears, f32
 * vectors) and contiguous layouts.
 * Errors: DLO_ERR_INVALID on null pointers, n_params < 1, ndim outside 1..4,
 * a non-positive extent, a negative stride, an unknown dtype, or
 * n_shards < 1. */
dlo_status dlo_plan_create(const dlo_param_desc* params, int32_t n_params,
                           int32_t n_shards, dlo_plan** out);
dlo_status dlo_plan_query(const dlo_plan* plan, dlo_plan_info* out);
dlo_status dlo_plan_group(const dlo_plan* plan, int32_t group, dlo_group_info* out);
dlo_status dlo_plan_param(const dlo_plan* plan, int32_t param, dlo_param_info* out);

/* CPU flatten / pad / split ([B2] §2, the rank-r copy window).
 * param_src[p]: host pointer to parameter p's element [0,..,0]; its
 *   storage_numel elements are read from there in memory order (n_params
 *   entries, in plan order).
 * shard_dst[g * n_shards + r]: host buffer of at least shard_alloc_bytes for
 *   group g, shard r (pinned memory for the stream to use it; any memory is
 *   accepted here).  Each is fully written: the shard's elements, then zeros.
 * Errors: DLO_ERR_INVALID on null pointers. */
dlo_status dlo_shard_host(const dlo_plan* plan, const void* const* param_src,
                          void* const* shard_dst);

/* One copy of a prefetch, by offsets: `bytes` bytes of shard (group,
 * shard) from src_offset to dst_offset of the copy's target. */
typedef struct {
  int32_t group;
  int32_t shard;
  int64_t dst_offset;  /* bytes from the start of the target (slot or staging) */
  int64_t src_offset;  /* bytes from the start of the host shard, or (a
                          gather) from the start of the staging buffer */
  int64_t bytes;
} dlo_copy_piece;

typedef enum {
  DLO_PIECES_SLOT_FROM_SHARDS = 0,   /* DMA / copy kernel: host shards -> slot */
  DLO_PIECES_STAGING_FROM_SHARDS = 1,/* staged phase 1: host shards -> staging */
  DLO_PIECES_SLOT_FROM_STAGING = 2   /* staged phase 2: staging -> slot */
} dlo_pieces_phase;

/* Checks one prefetch's copies against the plan: the layout of [B2] §2
 * (shard r of group g holds the group's flat elements [r*S_g, (r+1)*S_g))
 * placed as all_gather_into_tensor places it (shard r at base_g +
 * r*shard_bytes_g of the slot; in staging at stage_base_g +
 * r*shard_alloc_bytes_g).  Every piece must
 *   - name a valid (group, shard) and move at least one byte;
 *   - read inside its shard: bytes [x, x+bytes) with 0 <= x and x+bytes <=
 *     shard_bytes (into a slot) or shard_alloc_bytes (into staging), where
 *     x = src_offset, or for a gather src_offset minus the shard's staging
 *     offset;
 *   - write exactly where those bytes belong in the target, and inside its
 *     target_bytes;
 * no two pieces may write the same byte, and every byte [0, shard_bytes) of
 * every shard must be copied.
 * bad (optional) receives the first failing piece's index, or -1 (a shard
 * not fully copied, or no failure).
 * Errors: DLO_ERR_INVALID on null pointers or an unknown phase;
 * DLO_ERR_STATE when a rule fails (dlo_last_error names the piece and the
 * rule). */
dlo_status dlo_check_pieces(const dlo_plan* plan, int32_t phase, const dlo_copy_piece* pieces,
                            int32_t n, int64_t target_bytes, int32_t* bad);
void dlo_plan_destroy(dlo_plan* plan);

/* ------------------------------------------------------------------------
 * One-shot reassembly ([B1] "Weight Sharding + AllGather" steps 1-2; [D5]
 * "AllGather path"): copies every shard of a block host->device into `dst`
 * laid out as a slot, on `stream`, with the given mode (AUTO means DMA here).
 * shard_ptrs: as in dlo_shard_host; each must be 16-byte aligned and hold
 *   shard_alloc_bytes (the kernel path reads whole 16-byte words).  The
 *   kernel path needs page-locked, device-mapped memory (cudaHostAlloc or
 *   cudaHostRegister with mapping); DLO_ERR_INVALID otherwise.
 * dst: device buffer of at least plan slot_bytes; 256-byte aligned.
 * Asynchronous; the shard memory must stay valid until the stream passes. */
dlo_status dlo_reassemble(const dlo_plan* plan, const void* const* shard_ptrs,
                          void* dst, int32_t mode, void* stream);

/* One-shot staged reassembly (the DLO_COPY_STAGED phases, [B2] §3): the
 * shards move host->device into `staging` by DMA on copy_stream, then a
 * device-to-device copy-and-reassemble kernel on gather_stream (which waits
 * for the first phase through an event) writes `dst` laid out as a slot.
 * shard_ptrs: as in dlo_reassemble (page-locked; mapping not needed).
 * staging: device buffer of at least plan staging_bytes, 256-byte aligned.
 * dst: device buffer of at least plan slot_bytes, 256-byte aligned.
 * copy_stream and gather_stream may be the same stream.  Asynchronous; the
 * shards and staging must stay valid until gather_stream passes.
 * Errors: DLO_ERR_INVALID on null or misaligned pointers or a staging
 * buffer smaller than staging_bytes; DLO_ERR_CUDA on a CUDA failure. */
dlo_status dlo_reassemble_staged(const dlo_plan* plan, const void* const* shard_ptrs,
                                 void* staging, int64_t staging_bytes, void* dst,
                                 void* copy_stream, void* gather_stream);

/* ------------------------------------------------------------------------
 * Synthetic DiT block (the block the stream feeds; the pages do not define
 * one).  x is the fp32 residual [batch*tokens, hidden], updated in place:
 *   h  = RMSNorm(x) * g1 * (1 + scale1) + shift1          (bf16)
 *   qkv = h Wqkv^T                                         (bf16, [.., 3d])
 *   o  = softmax(q k^T / sqrt(hd)) v per head, non-causal  (bf16)
 *   x += gate1 * (o Wo^T)
 *   h2 = RMSNorm(x) * g2 * (1 + scale2) + shift2
 *   x += gate2 * (GELU_tanh(h2 W1^T) W2^T)
 * Linear weights are [out, in] (nn.Linear layout), bf16; norm gains and
 * adaLN vectors are fp32 [hidden].  Accumulation is fp32.
 * ------------------------------------------------------------------------ */

typedef struct {
  int32_t batch;
  int32_t tokens;
  int32_t hidden;   /* multiple of 64 */
  int32_t heads;    /* hidden / heads must be 64 or 128 */
  int32_t mlp;      /* multiple of 64 */
  float eps;        /* RMSNorm epsilon */
  int32_t flags;    /* DLO_FWD_* below.  DLO_FWD_GRAPH: launch the block's
                       kernels as one cached CUDA graph (captured on first
                       use for this config, plan, weight base, x and
                       scratch); results are the same bits as direct
                       launches */
} dlo_dit_cfg;

/* dlo_dit_cfg.flags:
 *   DLO_FWD_GRAPH    launch the block's kernels as one cached CUDA graph;
 *   DLO_FWD_ROPE     rotary position embedding of q and k after the QKV linear
 *                    (checkpoint-shaped block): the head's values in pairs
 *                    (2i, 2i+1) rotated by p * 10000^(-2i/hd) for the token at
 *                    position p within its batch item (RoFormer's form);
 *   DLO_FWD_QK_NORM  per-head RMSNorm of q and k (eps = cfg eps) with the
 *                    plan's fp32 gains "attn.q_norm.weight" and
 *                    "attn.k_norm.weight" [hd], before the rotary embedding;
 *                    required exactly when the plan has those gains.
 * Biases ("attn.qkv.bias" [3d], "attn.out.bias" [d], "mlp.fc1.bias" [f],
 * "mlp.fc2.bias" [d], bf16) are added to the linears' outputs whenever the
 * plan has them (before the GELU and before the gates). */
enum { DLO_FWD_GRAPH = 1, DLO_FWD_ROPE = 2, DLO_FWD_QK_NORM = 4 };

/* Bytes of device scratch one block forward needs (bf16 h, qkv, V
 * transposed, o, u, and the fp32 workspace of the linears run as K slices:
 * every tile when there are fewer tiles than SMs, or only the tiles of a
 * short last wave).  The split choice depends on the device's SM count. */
size_t dlo_forward_scratch_bytes(const dlo_dit_cfg* cfg);

/* Number of kernel launches one dlo_forward (or dlo_forward_noalloc) makes
 * for this configuration — two norm launches, attention plus one merge
 * launch when the items of its last wave run as KV slices, and for each of
 * the four linears (QKV, out-projection, fc1, fc2) one GEMM plus one ordered
 * reduction when some of its tiles run as K slices (the splits depend on the
 * current device's SM count; 152 when none is visible) — or 0 for an
 * invalid configuration.  Launches nothing. */
int32_t dlo_forward_launches(const dlo_dit_cfg* cfg);

/* One block forward with weights at `block_base`, laid out as a slot of
 * `plan` (the plan's parameter names must be the DiT block's: norm1.weight,
 * ada1.shift, ada1.scale, ada1.gate, attn.qkv.weight, attn.out.weight,
 * norm2.weight, ada2.shift, ada2.scale, ada2.gate, mlp.fc1.weight,
 * mlp.fc2.weight).  Used for the all-resident reference run; the streamed
 * path calls the same kernels through dlo_block_forward.
 * x: device fp32 [batch*tokens*hidden], 16-byte aligned, updated in place.
 * scratch: device, >= dlo_forward_scratch_bytes, 256-byte aligned.
 * Errors: DLO_ERR_INVALID on shapes the kernels do not support, a plan
 * without DiT roles or with mismatched shapes; DLO_ERR_NOMEM if scratch is
 * too small. */
dlo_status dlo_forward(const dlo_dit_cfg* cfg, const dlo_plan* plan,
                       const void* block_base, float* x, void* scratch,
                       size_t scratch_bytes, void* stream);

/* dlo_forward without a caller scratch buffer, for callers that cannot
 * allocate device memory: serving loops that must not allocate once warm
 * (cudaMalloc/cudaFree can synchronise the device and stall every stream),
 * and hosts whose device memory belongs to another allocator with a fixed
 * budget.  The pages have no counterpart of this call; it is an addition
 * of this library.
 * Scratch comes from a 32 MiB array in the library's own device memory
 * (a file-scope __device__ array, held by every GPU that loads the library
 * until the process exits).  A shape whose scratch
 * (dlo_forward_scratch_bytes) exceeds 32 MiB is rejected with
 * DLO_ERR_NOMEM.  The call allocates nothing: no cudaMalloc/cudaFree, no
 * graph instantiation (the block's kernels are launched directly, whatever
 * cfg->flags says).
 * The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress) with that device current; make that first call
 * before any stream capture.  Every call on a device shares the one array,
 * which keeps the last call's contents (the forward needs none of it to
 * start at zero): calls whose work overlaps on the GPU (other streams, or
 * other threads) race on it and must be serialised by the caller.
 * Arguments and errors are those of dlo_forward. */
dlo_status dlo_forward_noalloc(const dlo_dit_cfg* cfg, const dlo_plan* plan,
                               const void* block_base, float* x, void* stream);

/* Single steps of the block, for per-kernel checks (device pointers):
 *   rmsnorm_mod: h = bf16(x / sqrt(mean(x^2)+eps) * g * (1+scale) + shift)
 *   linear:      out = epilogue(a W^T + bias), a bf16 [M,K], W bf16 [N,K],
 *                bias bf16 [N] or null (none);
 *                epilogue 0: out bf16 [M,N] = acc
 *                         1: out bf16 [M,N] = GELU_tanh(acc)
 *                         2: out fp32 [M,N] += gate[N] * acc  (in place)
 *                K and N multiples of 8; pointers 16-byte aligned.
 *                workspace (device, may be null): when the output has too
 *                few 128x256 tiles to fill the GPU — or its tiles leave a
 *                last wave of at most half the SMs, for that wave's tiles
 *                only — K is split into slices computed in parallel into
 *                fp32 partials in the workspace, then summed in slice order
 *                (deterministic) by a second kernel that applies the
 *                epilogue; this needs dlo_op_linear_workspace_bytes(M, N, K,
 *                epilogue) bytes (0: the shape does not split).  Without
 *                enough workspace the linear runs unsplit.
 *   attention:   o bf16 [batch*tokens, d] from qkv bf16 [batch*tokens, 3d];
 *                scratch (device, 16-byte aligned) holds V transposed and,
 *                when the (batch, head, query group) items leave a last
 *                wave of at most half the SMs, the fp32 partial results of
 *                that wave's items split into KV slices (merged in slice
 *                order by a second kernel):
 *                dlo_op_attention_scratch_bytes(batch, tokens, d) bytes
 *                (inside dlo_forward the QKV linear writes V transposed
 *                directly).
 *   qk_norm_rope: in place on the q and k columns of qkv bf16
 *                [batch*tokens, 3d] (v untouched), per row and head of hd =
 *                d/heads (64 or 128): RMSNorm over the head with gains
 *                gq / gk fp32 [hd] (both null: none), then rotary embedding
 *                with base rope_base (0: none) as DLO_FWD_ROPE describes;
 *                pointers 16-byte aligned.  The angle is formed in fp32. */
dlo_status dlo_op_rmsnorm_mod(const float* x, int64_t rows, int64_t d,
                              const float* g, const float* shift,
                              const float* scale, float eps, uint16_t* h,
                              void* stream);
size_t dlo_op_linear_workspace_bytes(int64_t M, int64_t N, int64_t K, int32_t epilogue);
dlo_status dlo_op_linear(const uint16_t* a, int64_t M, int64_t K,
                         const uint16_t* w, int64_t N, int32_t epilogue,
                         void* out, const float* gate, const uint16_t* bias,
                         void* workspace, size_t workspace_bytes, void* stream);
size_t dlo_op_attention_scratch_bytes(int64_t batch, int64_t tokens, int64_t d);
dlo_status dlo_op_attention(const uint16_t* qkv, int64_t batch, int64_t tokens,
                            int64_t d, int64_t heads, uint16_t* o, void* scratch,
                            size_t scratch_bytes, void* stream);
dlo_status dlo_op_qk_norm_rope(uint16_t* qkv, int64_t batch, int64_t tokens,
                               int64_t d, int64_t heads, const float* gq,
                               const float* gk, float eps, float rope_base,
                               void* stream);

/* Which GEMM kernel runs the linears (a tuning and test switch; the
 * product of a linear is the same operation either way).  The linears run
 * either on single CTAs in 128 x 256 output tiles (with the K splits
 * described under dlo_op_linear) or unsplit on pairs of CTAs in 256 x 256
 * tiles, each CTA of a pair loading half of both operand tiles for one
 * tcgen05 MMA over the two SMs (cta_group::2).
 * mode: -1 (default) by shape: pairs when they fill at least one wave
 *       and an estimate of the two kernels' time (whole waves of pairs
 *       against the one-CTA kernel's waves plus the reduction of a split
 *       last wave) favours them; 0 never; 1 pairs for every linear.
 * Process-wide; takes effect for linears enqueued afterwards (a block
 * forward graph already captured keeps the kernels it was captured with).
 * The split workspace sizes (dlo_op_linear_workspace_bytes,
 * dlo_forward_scratch_bytes) and dlo_forward_launches follow the mode.
 * DLO_ERR_INVALID for another mode. */
dlo_status dlo_set_gemm_pair_mode(int32_t mode);
/* 1 if dlo_op_linear (and the block forward) runs a linear of this shape on
 * CTA pairs under the current mode on this GPU, else 0 (also for empty or
 * negative extents). */
int32_t dlo_op_linear_on_pairs(int64_t M, int64_t N, int64_t K, int32_t epilogue);

/* ------------------------------------------------------------------------
 * Engine: two slots, the hook schedule, events ([B1] "Double-Buffer Memory
 * Bound", "Slot Tracking: i%2 + Dynamic Correction"; [B2] §3; [D5]
 * "AllGather path").
 * ------------------------------------------------------------------------ */

/* ------------------------------------------------------------------------
 * Registered host ranges ([D5] "Registered mmap transport"): page-locks
 * complete host ranges (for example a read-only checkpoint mapping) so that
 * the rank-local path can copy tensor views straight from them into the
 * slots, without the two host staging slots.
 * ptrs[i], bytes[i]: n ranges; each is widened to whole pages, and ranges
 *   that then share pages are merged (a page is registered once); the
 *   merged ranges are registered in address order.
 * flags: 1 = the ranges are read-only (cudaHostRegisterReadOnly).
 * limit_bytes: > 0 caps the page-aligned total; over it nothing is
 *   registered and DLO_ERR_NOMEM is returned (the caller keeps staging).
 * All or nothing: on a failure the ranges registered by this call are
 * unregistered again and the status is DLO_ERR_CUDA; if an unregistration
 * fails too, DLO_ERR_PARTIAL (those mappings must not be closed).
 * *registered_bytes (may be null) receives the page-aligned total on
 * success.  Unregistering is the caller's, with dlo_host_unregister_ranges
 * (same ptrs/bytes); it unregisters every range and reports the first
 * failure (retryable). */
dlo_status dlo_host_register_ranges(const void* const* ptrs, const int64_t* bytes, int32_t n,
                                    int32_t flags, int64_t limit_bytes,
                                    int64_t* registered_bytes);
dlo_status dlo_host_unregister_ranges(const void* const* ptrs, const int64_t* bytes, int32_t n);

/* Test hook: replaces the CUDA registration calls used by the two
 * functions above with fakes (enable = 1): the fake register fails on its
 * call number fail_register_at (0-based; -1: never), the fake unregister on
 * call number fail_unregister_at.  Each fake call is logged; *n_calls and
 * log[] (capacity cap) receive entries of +(i+1) for "register range i" and
 * -(i+1) for "unregister range i" (i: index among the merged, address-ordered
 * page ranges).  enable = 0 restores the real calls.
 * Touches no GPU; for host-side tests of the all-or-nothing contract. */
dlo_status dlo_debug_fake_host_register(int32_t enable, int32_t fail_register_at,
                                        int32_t fail_unregister_at);
dlo_status dlo_debug_fake_host_register_log(int32_t* log, int32_t cap, int32_t* n_calls);

typedef struct dlo_engine dlo_engine;

typedef struct {
  int32_t n_blocks;       /* blocks per pass (hooks), >= 1 */
  void* slot[2];          /* device buffers, 256-byte aligned, caller-owned */
  int64_t slot_bytes;     /* capacity of each slot */
  void* compute_stream;   /* cudaStream_t for block forwards */
  void* copy_stream;      /* cudaStream_t for prefetches (must differ) */
  int32_t copy_mode;      /* dlo_copy_mode */
  int32_t copy_ctas;      /* CTAs of the copy kernel; 0 = default (152) */
  int32_t timing;         /* 1: bracket every prefetch with timing events */
  int32_t dma_streams;    /* DMA fan-out: the (group, shard) copies of one
                             prefetch are spread over this many library-owned
                             streams forked from the copy stream and joined
                             back before the ready event; 0 = default (1:
                             every copy on the copy stream, which measured
                             faster on GB300 than spreading them) */
  void* staging[2];       /* DLO_COPY_STAGED only: device staging buffers,
                             256-byte aligned, caller-owned; staging[x] serves
                             the prefetches into slot x.  Null otherwise. */
  int64_t staging_bytes;  /* capacity of each staging buffer (>= every
                             registered block's plan staging_bytes) */
  void* gather_stream;    /* DLO_COPY_STAGED only: cudaStream_t of the
                             device-to-device phase; differs from the other
                             two streams.  The H2D into staging[x] waits only
                             for the gather that last read staging[x]; the
                             gather waits for the H2D and for the slot's free
                             event, and records the slot's ready event. */
  void* host_staging[2];  /* rank-local source blocks only (see
                             dlo_register_block_source): two page-locked
                             host buffers, caller-owned, into which CPU
                             threads pack a block before its DMA; host
                             staging x serves the prefetches into slot x.
                             Null when unused. */
  int64_t host_staging_bytes; /* capacity of each (>= a packed block's
                             slot_bytes) */
  int32_t pack_threads;   /* CPU threads that pack a block (0 = 4) */
  int32_t two_copy_streams;/* 0 (default): every prefetch on copy_stream,
                             as the pages draw it; 1: prefetches into slot 1
                             on a second, library-owned stream, so that the
                             copies of consecutive blocks may overlap at their
                             ends (each still waits for its slot's free
                             event).  Measured on GB300 with one H2D link: no
                             gain, the copy engines run them one at a time */
  int32_t log_capacity;   /* entries kept by the schedule log (one per
                             forward) and by the timing record (one per
                             prefetch, timing = 1): the newest ones; once full
                             each new entry overwrites the oldest, which is
                             counted as dropped, so a serving loop of any
                             length holds constant memory.  0 = 65536;
                             at most 2^24 */
  int32_t poison;         /* debugging: 1 = after each forward, overwrite the
                             slot it read with the byte 0xA5 on the compute
                             stream, before the slot's free event, so that a
                             forward reading a slot the schedule has
                             released, or one not yet refilled, sees garbage
                             rather than a plausible stale block.  Costs one
                             device memset of the slot per forward; 0 (the
                             default) = off */
  int32_t checks;         /* debugging: 1 = every prefetch of a block
                             registered by shards first lists its copies
                             without issuing them (DMA pieces, the rows of
                             2-D copies, copy-kernel segments, staged H2D and
                             gather) and checks their offsets with
                             dlo_check_pieces; a prefetch that fails is not
                             issued and returns DLO_ERR_STATE.  dlo_param_view
                             also checks that the view lies inside its
                             group's gathered elements and the slot.  Host
                             work only (a few microseconds a prefetch);
                             0 (the default) = off */
} dlo_engine_desc;

typedef struct {
  int32_t k;                  /* global forward index */
  int32_t block;
  int32_t read_slot;
  int32_t prefetch_block;
  int32_t prefetch_slot;
  int32_t waits_on_free_of_k; /* forward whose free event the prefetch waited on; -1: none */
  int32_t copy_mode;          /* mode used for the prefetch */
} dlo_sched_event;

/* Creates an engine.  Each hook i starts with current_slot = i % 2 and no
 * prefetched slot; hook 0's predecessor is hook n_blocks-1 (circular).
 * Errors: DLO_ERR_INVALID on null/misaligned slots, equal streams,
 * n_blocks < 1; DLO_ERR_CUDA if events cannot be created. */
dlo_status dlo_engine_create(const dlo_engine_desc* desc, dlo_engine** out);

/* Registers block `block` (0 <= block < n_blocks) with its plan and shard
 * pointers (shard_ptrs[g * n_shards + r], host, pinned, 16-byte aligned,
 * shard_alloc_bytes each; borrowed until dlo_engine_destroy).  The plan is
 * borrowed too.  Several blocks may share one plan and one set of shards.
 * Errors: DLO_ERR_INVALID (range, plan larger than a slot, pointer not
 * pinned/mapped or misaligned), DLO_ERR_STATE (already registered). */
dlo_status dlo_register_block(dlo_engine* e, int32_t block, const dlo_plan* plan,
                              const void* const* shard_ptrs);

/* Points registered `block` at a new copy of its shards (same plan; the
 * pointers obey dlo_register_block's rules), for a caller that moves a
 * block's host memory while the stream runs — for example off host ranges
 * that have turned slow for the GPU to read.  First waits (host side,
 * bounded by timeout_ms) until every copy already enqueued from the old
 * shards has completed, so that the caller may reuse the old memory once
 * the call returns; later prefetches read the new shards.  Several engine
 * blocks registered with the same shards are replaced one by one.
 * The pages have no counterpart: they load every shard once ([B2] §2);
 * their nearest step is the drain of in-flight host-to-device copies
 * before host memory is released ([D5] "Lease ownership").
 * Errors: DLO_ERR_INVALID (range, pointers), DLO_ERR_STATE (the block is
 * not registered with shards), DLO_ERR_TIMEOUT (a pending copy did not
 * finish in time; nothing is changed). */
dlo_status dlo_replace_block_shards(dlo_engine* e, int32_t block,
                                    const void* const* shard_ptrs, int32_t timeout_ms);

/* Rank-local source blocks ([D5] "Rank-local path without DLO AllGather"):
 * registers `block` by the host addresses of its parameters instead of by
 * shards.  The plan must have n_shards = 1 (no sharding on this path).
 * param_src[p]: parameter p's element [0,..,0] in any host memory (pageable
 *   runtime tensors, a checkpoint mapping); storage_numel elements are read
 *   in memory order.  Borrowed until the engine is destroyed.
 * If every parameter lies in page-locked memory (for example ranges
 * registered with dlo_host_register_ranges), each prefetch copies every
 * parameter straight into its slot offset ("Registered mmap transport").
 * Otherwise each prefetch into slot x first waits for the DMA that last read
 * host staging x, packs the parameters there on pack_threads CPU threads (in
 * the calling thread, which returns once the pack is done), then moves the
 * packed block with one DMA ("two bounded pinned host staging slots");
 * the engine's host staging buffers are then required.
 * Errors: DLO_ERR_INVALID on bad arguments, n_shards != 1, a block too
 * large for the slots or host staging, or no host staging for a pageable
 * source; DLO_ERR_STATE if the block is registered already. */
dlo_status dlo_register_block_source(dlo_engine* e, int32_t block, const dlo_plan* plan,
                                     const void* const* param_src);

/* Enqueues a prefetch of `block` into `slot` on the copy stream: the copy
 * stream waits for the free event of the forward that last read `slot`,
 * copies and reassembles, then records the slot's ready event.  This is the
 * setup prefetch (block 0 into slot 0) before the first forward; the hook
 * issues all later prefetches itself.
 * Errors: DLO_ERR_INVALID (range), DLO_ERR_STATE (block unregistered). */
dlo_status dlo_prefetch(dlo_engine* e, int32_t block, int32_t slot);

/* Makes the compute stream wait for the ready event of the slot holding
 * `block` (non-blocking on the host).  During that block's forward this is
 * the slot its hook picked; otherwise the slot filled with it last (with a
 * one-block pass both slots hold the block, and the newer copy is the one
 * the next forward reads).  The same slot resolves dlo_wait_host and
 * dlo_param_view.  DLO_ERR_STATE if no slot holds it. */
dlo_status dlo_wait(dlo_engine* e, int32_t block);

/* Host-side poll of the same event, bounded by timeout_ms; DLO_ERR_TIMEOUT
 * when it runs out.  Never spins on the device. */
dlo_status dlo_wait_host(dlo_engine* e, int32_t block, int32_t timeout_ms);

/* Device pointer of parameter `param` of resident `block` (a view into the
 * slot, no copy; [B1] "Weight Sharding + AllGather" step 3).
 * DLO_ERR_STATE if no slot holds the block. */
dlo_status dlo_param_view(const dlo_engine* e, int32_t block, int32_t param,
                          void** dev_ptr);

/* The pre-forward hook of block `block`, which must be the next block of
 * the pass (global forward k -> block k mod n_blocks):
 *   1. adopt the previous hook's prefetched slot, if it has one;
 *   2. make the compute stream wait for that slot's ready event;
 *   3. prefetch block (block+1) mod n_blocks into the other slot (circular
 *      tail->head wrap), after the free event of that slot's last reader;
 *   4. record the prefetched slot.
 * Writes the slot the forward must read to *slot_out (may be null).
 * Errors: DLO_ERR_STATE if `block` is not the next block, if the slot does
 * not hold it, or if a post_forward is missing. */
dlo_status dlo_pre_forward(dlo_engine* e, int32_t block, int32_t* slot_out);

/* Records the free event of the slot just read, on the compute stream. */
dlo_status dlo_post_forward(dlo_engine* e, int32_t block);

/* pre_forward + dlo_forward on the slot + post_forward. */
dlo_status dlo_block_forward(dlo_engine* e, int32_t block, const dlo_dit_cfg* cfg,
                             float* x, void* scratch, size_t scratch_bytes);

/* Copies the newest min(cap, kept) entries of the schedule log (one per
 * forward, oldest first) to buf; *n_out = the number of entries kept (at
 * most desc.log_capacity; older ones are counted in
 * dlo_engine_stats.log_dropped).  cap = 0 with a null buf queries *n_out. */
dlo_status dlo_schedule_log(const dlo_engine* e, dlo_sched_event* buf,
                            int32_t cap, int32_t* n_out);

/* Engine counters.  copy_ms[i] / copy_bytes[i]: elapsed time and bytes of
 * the i-th timed prefetch (only with desc.timing = 1; synchronises on the
 * events it reads).  chosen_mode: the mode AUTO settled on (or the fixed
 * mode; DLO_COPY_AUTO while undecided); n_kernel_prefetches counts
 * copy-kernel launches.  AUTO races the two modes on the quantity that
 * matters, the compute stream's time per block forward while the next
 * block streams in.  With n = n_blocks, four windows of 6 forwards start at
 * forward n+2 (after one full pass, so first-touch costs are excluded):
 * the prefetches issued in windows 1 and 3 use DMA, in windows 2 and 4 the
 * copy kernel; race_dma_us / race_kernel_us are each mode's better
 * window's mean interval between consecutive free events (0 until
 * measured; -1 if the events could not be timed, in which case DMA is
 * chosen).  The timing record keeps the newest desc.log_capacity prefetches:
 * copy_times and copy_spans report those, oldest first. */
typedef struct {
  int32_t chosen_mode;
  int32_t n_forwards;
  int32_t n_prefetches;
  int32_t n_kernel_prefetches;
  double race_dma_us;
  double race_kernel_us;
  int32_t n_direct_prefetches; /* source blocks copied straight from
                                  page-locked parameters */
  int32_t n_packed_prefetches; /* source blocks packed into host staging */
  double pack_ms;              /* host time spent packing (waits included) */
  int32_t n_copy_kernel_launches; /* copy-kernel launches of all prefetches:
                                  KERNEL prefetches, DMA prefetches' small
                                  groups, STAGED gathers */
  int64_t log_dropped;         /* schedule-log entries overwritten (full ring) */
  int64_t timed_dropped;       /* timing entries overwritten (full ring) */
  int64_t checked_pieces;      /* copies checked before issue (desc.checks) */
} dlo_engine_stats;
dlo_status dlo_engine_query(dlo_engine* e, dlo_engine_stats* out);
dlo_status dlo_engine_copy_times(dlo_engine* e, float* copy_ms, int64_t* copy_bytes,
                                 int32_t cap, int32_t* n_out);
/* With timing = 1: each kept prefetch's start and end (ms) on one clock,
 * counted from the oldest kept prefetch's start, for the first `cap` of
 * them; *n_out = how many are kept.  Prefetches into the two slots may overlap
 * (two copy streams), so the copy engines' busy time is the union of these
 * intervals, not the sum of copy_times.  Blocks until the spans' end events
 * have completed. */
dlo_status dlo_engine_copy_spans(dlo_engine* e, float* start_ms, float* end_ms,
                                 int32_t cap, int32_t* n_out);

/* One timed prefetch (desc.timing = 1). */
typedef struct {
  int64_t seq;          /* 0, 1, 2, ...: the engine's n-th timed prefetch */
  int32_t block;        /* block copied */
  int32_t slot;         /* slot written */
  float copy_ms;        /* time between the events around its copies */
  int64_t bytes;        /* bytes moved */
} dlo_copy_record;

/* Incremental, non-blocking read of the timing record ([B1] "Overlap
 * Analysis" reads prefetch against compute time per block from the run's
 * log; this is that record, per prefetch): copies to buf, in
 * order, up to `cap` records of timed prefetches with seq >= since whose
 * copies have completed, stopping at the first one still in flight;
 * *n_out = how many, *next = the seq to pass as `since` next time.  Records
 * older than the ring kept (desc.log_capacity) are skipped.  A monitor in a
 * serving loop calls this between steps without waiting on the GPU.
 * Errors: DLO_ERR_INVALID (null n_out/next, or cap > 0 with a null buf). */
dlo_status dlo_engine_copy_log(dlo_engine* e, int64_t since, dlo_copy_record* buf, int32_t cap,
                               int32_t* n_out, int64_t* next);

/* Waits (host side, bounded by timeout_ms) for both streams' enqueued
 * engine work, then releases the engine's events.  The caller's buffers are
 * untouched.  Returns DLO_ERR_TIMEOUT (and keeps the engine) if the work
 * does not finish in time.  A null engine is accepted. */
dlo_status dlo_engine_destroy(dlo_engine* e, int32_t timeout_ms);

/* Device-side status of the library's kernels: every spin-wait inside a
 * kernel is bounded; a wait that runs out records a code here and the
 * kernel returns early.  Reads and clears the word (synchronises the
 * device).  *code = 0 means no wait ran out. */
dlo_status dlo_kernel_status(int32_t* code);

/* Fail-closed check of the kernels' bounded device waits (the pages' "fail
 * closed" rule: [B1] "Fail-Closed Design"; [B2] "Validation Results", a
 * partial wave that times out fails closed).  Launches one small library
 * kernel (one CTA, synchronously, on the legacy default stream) whose
 * thread waits, with the wait routine every kernel of the library uses
 * (spin = 1: the spinning form of MMA issuers, 0: the suspending form),
 * on an mbarrier phase that no thread completes, with limit_ns in place of
 * the kernels' 4 s; if abort_ns > 0 a second warp raises the CTA's abort
 * flag after abort_ns instead, the path by which one role of a kernel stops
 * the others.  The wait gives up, the kernel records its code in the
 * device error word and returns; the context stays usable.
 * *elapsed_ns: how long the wait ran (device clock); *code: the recorded
 * code (7 = timed out, 6 = aborted), which is also cleared from the word.
 * Returns DLO_ERR_TIMEOUT when the wait gave up (the expected outcome),
 * DLO_ERR_INVALID for limits outside 0..2 s.  Allocates nothing. */
dlo_status dlo_debug_wait_probe(int32_t spin, int64_t limit_ns, int64_t abort_ns,
                                int64_t* elapsed_ns, int32_t* code);

/* Launch overlap of the block forward's kernels (process-wide): with it,
 * every kernel of a block after the first is launched with programmatic
 * stream serialization, so that its CTAs may be scheduled and do their
 * set-up (barriers, tensor memory, descriptor prefetch) while the previous
 * kernel drains; each waits for that kernel's completion before it touches
 * memory, so results are bit for bit those without.  1 always, 0 never,
 * -1 (default) for blocks below 1e11 FLOPs only (measured on GB300: 2% off
 * a 1024-hidden, 1024-token block's forward; 1.5% slower on the
 * 6144-hidden, 8192-token one).  The forward's cached CUDA graphs are keyed
 * on the resulting choice.  The pages have no counterpart (their forward is
 * a framework's; [B2] "Validation Results" counts its Python dispatch and
 * stream switches as overhead, which this launch path and the graphs
 * address).  DLO_ERR_INVALID unless -1, 0 or 1. */
dlo_status dlo_set_launch_overlap(int32_t on);

/* Message of the last failed call on this thread ("" if none). */
const char* dlo_last_error(void);

/* Library version, for diagnostics. */
const char* dlo_version(void);

#ifdef __cplusplus
}
#endif
#endif /* DLO_H_ */
