/*
 * mla_draft.h -- C ABI of the MLA (Multi-head Latent Attention) draft-layer
 * forward for NVIDIA GB300 (sm_103a).
 *
 * What the layer computes (sources are web pages, cited by title/section):
 *  - "MLA (Multi-Head Latent Attention)" blog, DeepseekV2MLAAttention.__init__
 *    and MultiHeadLatentAttentionWrapper.forward: optional low-rank query
 *    (fused_qkv_a_proj -> q_a_layernorm -> q_b_proj, or q_proj without
 *    q_lora_rank), the shared compressed KV latent (kv_a_proj_with_mqa ->
 *    kv_a_layernorm), partial RoPE on qk_rope_head_dim, kv_b_proj expansion,
 *    o_proj.
 *  - same blog, do_kv_cache_update / concat_and_cache_mla and
 *    get_kv_cache_shape: the latent cache [num_pages, page_size,
 *    kv_lora_rank + qk_rope_head_dim], one entry [kv_c_normed | k_pe] per
 *    token, written by slot index.
 *  - same blog, forward_impl (MQA branch) and forward_mqa: attention in the
 *    latent space (q_nope @ W_UK, scores against [c | k_pe], W_UV up-proj).
 *  - "Add config-selectable MLA draft attention" (SpecForge PR #758),
 *    Summary/Structure: DFlash-family target-context injection, full/sliding
 *    masks, zeroing of fully masked queries, optional output gate, NeoX or
 *    interleaved rotation; dimension validation once at init.
 *  - "extract GQA/MLA attention into reusable layers" (SpecForge PR #1026),
 *    Modifications: masks by logical position; empty queries zeroed before
 *    o_proj.
 *
 * Conventions for every entry point
 *  - Pointers named "device" are CUDA device pointers (cudaMalloc / torch),
 *    "host" pointers are CPU memory.  The library never allocates device
 *    memory: weights, arena, cache, workspace and outputs belong to the
 *    caller.  The library owns only the host-side handle.
 *  - Weights use torch.nn.Linear layout W[out, in], row-major, contiguous, of
 *    the config's dtype (bf16 or fp32).  Hidden states are row-major
 *    [tokens, hidden_size] of the same dtype; so is the cache.
 *  - `stream` is a cudaStream_t (NULL = legacy default stream).  append and
 *    forward only enqueue work: no host synchronisation, no allocation.
 *  - Errors: host-side validation returns a status and never aborts; the
 *    message is available from mla_last_error().  Index errors found on the
 *    device (slot, page or position out of range) skip the offending access
 *    and set a bit in a device status word read by mla_get_device_status().
 *  - Devices: one GPU per process.  A handle works on the device that was
 *    current at mla_draft_init, which must be current for every call; the
 *    library keeps per-process launch settings (kernel shared-memory limits,
 *    the SM count and cluster occupancy) taken from the first device it
 *    runs on.  The multi-GPU model is one process per GPU.
 */
#ifndef MLA_DRAFT_H
#define MLA_DRAFT_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int32_t mla_status_t;
enum {
  MLA_OK = 0,
  MLA_ERR_INVALID_ARG = 1,   /* null pointer, bad size, inconsistent dims    */
  MLA_ERR_UNSUPPORTED = 2,   /* valid dims this build has no kernel for       */
  MLA_ERR_CUDA = 3,          /* a CUDA runtime/driver call failed             */
  MLA_ERR_DEVICE_CHECK = 4,  /* the device reported an index error            */
  MLA_ERR_TIMEOUT = 5        /* a bounded device wait expired                 */
};

enum { MLA_BF16 = 0, MLA_FP32 = 1 };              /* mla_config_t.dtype */
enum { MLA_ROPE_NEOX = 0, MLA_ROPE_INTERLEAVED = 1 }; /* mla_config_t.rope */

/* Bits of the device status word (mla_get_device_status). */
enum {
  MLA_DEV_BAD_SLOT = 1,      /* slot_mapping entry outside the cache          */
  MLA_DEV_BAD_POSITION = 2,  /* position < 0 or >= max_position               */
  MLA_DEV_BAD_PAGE = 4,      /* block_table entry outside [0, num_pages)      */
  MLA_DEV_TIMEOUT = 8,       /* a bounded mbarrier wait gave up               */
  MLA_DEV_BAD_LENGTH = 16,   /* kv_len < 0 or > max_pages * page_size         */
  MLA_DEV_BAD_WINDOW = 32    /* window < 0 (the block's rows are zeroed)      */
};

/* Intermediate tensors the forward leaves in its workspace
 * (mla_forward_workspace_offset). */
enum { MLA_WS_Q_ABS = 0, MLA_WS_O_LAT = 1, MLA_WS_O = 2 };

/* Layer configuration.  Structural dims follow the HF DeepSeek-V2/V3 fields;
 * q_lora_rank == 0 selects the non-low-rank path (q_proj +
 * kv_a_proj_with_mqa).  softmax_scale == 0 means 1/sqrt(qk_nope + qk_rope).
 * max_position bounds the RoPE table built at init. */
typedef struct {
  int32_t hidden_size, num_heads, q_lora_rank, kv_lora_rank;
  int32_t qk_nope_head_dim, qk_rope_head_dim, v_head_dim;
  int32_t rope;              /* MLA_ROPE_NEOX | MLA_ROPE_INTERLEAVED          */
  int32_t use_output_gate;   /* 0/1: o *= sigmoid(x @ gate_proj^T)            */
  int32_t dtype;             /* MLA_BF16 | MLA_FP32                           */
  int32_t page_size;         /* tokens per cache page                         */
  int32_t max_position;      /* positions must lie in [0, max_position)       */
  double rope_theta, rms_norm_eps, softmax_scale;
} mla_config_t;

/* Device pointers to the layer's parameters, read only inside mla_draft_init
 * (not retained).  Unused fields are NULL. */
typedef struct {
  const void *fused_qkv_a_proj;    /* [q_lora_rank + kv_lora_rank + qk_rope, D]  (q_lora_rank > 0) */
  const void *q_a_layernorm;       /* [q_lora_rank]                               (q_lora_rank > 0) */
  const void *q_b_proj;            /* [H * (qk_nope + qk_rope), q_lora_rank]      (q_lora_rank > 0) */
  const void *q_proj;              /* [H * (qk_nope + qk_rope), D]                (q_lora_rank == 0) */
  const void *kv_a_proj_with_mqa;  /* [kv_lora_rank + qk_rope, D]                 (q_lora_rank == 0) */
  const void *kv_a_layernorm;      /* [kv_lora_rank]                                                */
  const void *kv_b_proj;           /* [H * (qk_nope + v_head), kv_lora_rank]                        */
  const void *gate_proj;           /* [H * v_head, D]                             (use_output_gate) */
  const void *o_proj;              /* [D, H * v_head]                                               */
} mla_weights_t;

/* Which keys each query block attends (device pointers).  Block b holds
 * queries b*block_len .. (b+1)*block_len-1.  Its key j (logical position j)
 * is the cache entry at page block_table[b*max_pages + j/page_size], row
 * j%page_size.  Key j is visible to query i of block b iff
 *   q_visible[i] != 0  &&  j < kv_len[b]  &&
 *   (window[b] == 0 || positions[i] - j < window[b]).
 * A query with no visible key produces an exact zero output row.  A negative
 * window is rejected on the device: MLA_DEV_BAD_WINDOW is set and the block's
 * rows see no key. */
typedef struct {
  int32_t num_blocks, block_len, max_pages, reserved;
  const int32_t *block_table;  /* [num_blocks, max_pages]                      */
  const int32_t *kv_len;       /* [num_blocks]                                 */
  const int32_t *window;       /* [num_blocks]; NULL = every block full        */
  const uint8_t *q_visible;    /* [num_blocks * block_len]; NULL = all visible */
  int32_t *vis_stats;          /* optional output [num_blocks*block_len, 3]:
                                  visible-key count, first and last visible
                                  key (-1 when none), as the kernel's own mask
                                  applied them; NULL = not written            */
} mla_attn_desc_t;

/* Blocks that share a context (MLA blog, forward_impl: the prefill path,
 * forward_mha with _compute_prefill_context, runs the expanded form when
 * many query rows meet one cached context).  Context c's blocks are
 * ctx_block_start[c] .. ctx_block_start[c+1]-1 (consecutive; the whole list
 * covers blocks 0 .. num_blocks-1).  Each block b of context c sees keys
 * 0 .. ctx_len[c]-1 as the context -- the same cache entries for all of c's
 * blocks, read through the table of block ctx_block_start[c] -- and keys
 * ctx_len[c] .. kv_len[b]-1 as its own, at most block_len of them
 * (kv_len[b] <= ctx_len[c] + block_len; a longer kv_len is reported on the
 * device as MLA_DEV_BAD_LENGTH and its extra keys are not seen).  The
 * visibility rule of mla_attn_desc_t applies unchanged. */
typedef struct {
  int32_t num_ctx;                 /* contexts, 1 .. num_blocks (else
                                      MLA_ERR_INVALID_ARG)                       */
  int32_t ctx_rows;                /* host: sum of ctx_len (keys of all contexts) */
  const int32_t *ctx_len;          /* device [num_ctx]                           */
  const int32_t *ctx_block_start;  /* device [num_ctx + 1]                       */
} mla_shared_ctx_t;

typedef struct mla_handle mla_handle_t;

/* ---- geometry (host only; no GPU needed) --------------------------------
 * MLA blog, MLAAttention.__init__ / get_kv_cache_shape: one cache entry is
 * kv_lora_rank + qk_rope_head_dim wide (576 for DeepSeek dims), one KV head;
 * MLAAttentionSpec.real_page_size_bytes: page bytes = page_size * 1 *
 * entry * dtype size.  Return 0 for a NULL or inconsistent config. */
int32_t mla_cache_entry_dim(const mla_config_t *cfg);
size_t mla_cache_page_bytes(const mla_config_t *cfg);

/* Bytes of the derived-weight arena mla_draft_init fills (0 = invalid cfg). */
size_t mla_weight_arena_bytes(const mla_config_t *cfg);

/* Validate `cfg` (returns MLA_ERR_INVALID_ARG / MLA_ERR_UNSUPPORTED with a
 * message), re-lay the weights out into the caller's device `arena`
 * (>= mla_weight_arena_bytes): W_UK / W_UV split out of kv_b_proj (MLA blog,
 * forward_impl: W_UK_T and _v_up_proj), the A-projection rows ordered
 * [kv | q | gate], a RoPE cos/sin table computed in fp64 on the host, and the
 * device status word.  Synchronises `stream` before returning; `w` is not
 * retained.  On success *out receives a handle owned by the caller (free with
 * mla_draft_destroy).  One handle serves one stream at a time. */
mla_status_t mla_draft_init(const mla_config_t *cfg, const mla_weights_t *w,
                            void *arena, size_t arena_bytes, void *stream,
                            mla_handle_t **out);

/* Device scratch needed by one append of n tokens / one forward of
 * num_tokens block tokens. */
size_t mla_append_workspace_bytes(const mla_handle_t *h, int32_t n);
size_t mla_forward_workspace_bytes(const mla_handle_t *h, int32_t num_tokens);

/* Latent-cache append (target-context injection, PR #758; MLA blog,
 * do_kv_cache_update): for each of the n tokens,
 *   kv = hidden[t] @ W_kva^T            (W_kva = last kv_lora_rank+qk_rope rows
 *                                         of fused_qkv_a_proj, or
 *                                         kv_a_proj_with_mqa)
 *   cache[slot_mapping[t]] = [RMSNorm(kv[:r]) * kv_a_layernorm |
 *                             RoPE(kv[r:], positions[t])]
 * hidden: device [n, hidden_size]; positions: device int32 [n];
 * slot_mapping: device int64 [n], slot = page * page_size + row;
 * cache: device [num_pages, page_size, entry].  n == 0 is a no-op. */
mla_status_t mla_latent_cache_append(mla_handle_t *h, const void *hidden,
                                     const int32_t *positions,
                                     const int64_t *slot_mapping, int32_t n,
                                     void *cache, int32_t num_pages,
                                     void *workspace, size_t workspace_bytes,
                                     void *stream);

/* Draft-layer forward for desc->num_blocks blocks of desc->block_len tokens
 * (MLA blog, wrapper forward + forward_impl MQA branch; PR #758 masks, gate):
 *   q = rope(q_b_proj(RMSNorm(q_c)))  (or q_proj), absorbed with W_UK;
 *   latent attention over the cache keys each block sees (mla_attn_desc_t);
 *   o = W_UV * latent output, optionally * sigmoid(hidden @ gate_proj^T);
 *   out = o @ o_proj^T.
 * hidden: device [nb*T, hidden_size]; positions: device int32 [nb*T];
 * block_slot_mapping: device int64 [nb*T] -- when non-NULL the block's own
 * latents are written to the cache there before attending; when NULL they
 * must already be in the cache (mla_latent_cache_append).  out: device
 * [nb*T, hidden_size].  Fully masked query rows come out as exact +0.
 * Any block_len.  bf16 layers run the tensor-core kernels, which need
 * kv_lora_rank 512, qk_rope_head_dim 64, a page_size of 16, 32, 64 or a
 * multiple of 128, hidden_size, q_lora_rank, qk_nope_head_dim and
 * num_heads * v_head_dim multiples of 64; mla_draft_init rejects other bf16
 * shapes with MLA_ERR_UNSUPPORTED (the fp32 layer has no such limits).  The
 * workspace must be 256-byte aligned. */
mla_status_t mla_draft_forward(mla_handle_t *h, const void *hidden,
                               const int32_t *positions,
                               const int64_t *block_slot_mapping, void *cache,
                               int32_t num_pages, const mla_attn_desc_t *desc,
                               void *out, void *workspace,
                               size_t workspace_bytes, void *stream);

/* mla_draft_forward whose attention waits for an event.  Everything that
 * does not read the cache -- the projections, query RoPE and W_UK
 * absorption, and the block's own latents when block_slot_mapping is
 * non-NULL -- is enqueued on `stream` at once; before the attention, the
 * stream waits for `cache_ready` (a cudaEvent_t the caller recorded after
 * the cache writes the attention reads, typically mla_latent_cache_append
 * of the target context on another stream).  The block's projections then
 * run while the context is appended (the pages' draft reads the context
 * only through the attention's keys).  The two must write disjoint slots;
 * an append that needs a workspace needs its own.  cache_ready == NULL is
 * exactly mla_draft_forward.  Graph-capturable: recorded into a stream
 * capture, the event forks and joins the two streams.  Same arguments,
 * results and errors as mla_draft_forward otherwise. */
mla_status_t mla_draft_forward_after(mla_handle_t *h, const void *hidden,
                                     const int32_t *positions,
                                     const int64_t *block_slot_mapping, void *cache,
                                     int32_t num_pages, const mla_attn_desc_t *desc,
                                     void *out, void *workspace,
                                     size_t workspace_bytes, void *stream,
                                     void *cache_ready);

/* mla_draft_forward for blocks that share contexts (mla_shared_ctx_t), in
 * the expanded form when the layer allows it (bf16, kv_lora_rank 512,
 * qk_rope_head_dim 64, qk_nope_head_dim and v_head_dim 128, block_len <=
 * 128): each context's latents and each block's
 * own latents are expanded once by kv_b_proj into per-head k_nope and v
 * (MLA blog, forward_mha: kv_b_proj on the prefill context), the queries
 * keep q_nope and q_pe (no W_UK / W_UV absorption), and one attention runs
 * per (head, up to 128 / block_len blocks of a context): the context keys,
 * then the blocks' own keys as one more key tile, masked to each block's
 * own.  Other layers run mla_draft_forward.  Same results and errors as
 * mla_draft_forward, plus MLA_ERR_INVALID_ARG for a NULL context list or one
 * outside its contract (num_ctx not in 1 .. num_blocks, ctx_rows < 0); the
 * workspace (256-byte aligned, caller-owned) is
 * mla_forward_shared_workspace_bytes(h, num_tokens, ctx_rows) bytes, 0 for
 * a NULL handle or negative counts. */
size_t mla_forward_shared_workspace_bytes(const mla_handle_t *h, int32_t num_tokens,
                                          int32_t ctx_rows);
mla_status_t mla_draft_forward_shared(mla_handle_t *h, const void *hidden,
                                      const int32_t *positions,
                                      const int64_t *block_slot_mapping, void *cache,
                                      int32_t num_pages, const mla_attn_desc_t *desc,
                                      const mla_shared_ctx_t *ctx, void *out,
                                      void *workspace, size_t workspace_bytes,
                                      void *stream);

/* mla_draft_forward_shared whose attention waits for an event, as
 * mla_draft_forward_after: everything before the gather of the cache rows
 * is enqueued at once, then the stream waits for `cache_ready`. */
mla_status_t mla_draft_forward_shared_after(mla_handle_t *h, const void *hidden,
                                            const int32_t *positions,
                                            const int64_t *block_slot_mapping, void *cache,
                                            int32_t num_pages, const mla_attn_desc_t *desc,
                                            const mla_shared_ctx_t *ctx, void *out,
                                            void *workspace, size_t workspace_bytes,
                                            void *stream, void *cache_ready);

/* The attention step of mla_draft_forward_shared alone, on the intermediates
 * the last such call left in `workspace` (same handle, descriptor, context
 * list and token count): the queries' q_nope and q_pe, the gathered latent
 * rows and their kv_b_proj expansion, the gate.  It rewrites the workspace's
 * per-head output o (the input of o_proj) with the same values the forward
 * computed.  For timing and checking that step in isolation.
 * MLA_ERR_UNSUPPORTED when the layer does not take the expanded form,
 * MLA_ERR_INVALID_ARG for NULL pointers, a context list outside its contract
 * or a workspace smaller than mla_forward_shared_workspace_bytes(). */
mla_status_t mla_shared_attention(mla_handle_t *h, const int32_t *positions,
                                  const mla_attn_desc_t *desc, const mla_shared_ctx_t *ctx,
                                  void *workspace, size_t workspace_bytes, void *stream);

/* Allocation-free latent-cache append.  The pages have no counterpart: this
 * is a library convenience for callers that cannot allocate device memory
 * where they append (host callbacks, allocator hooks, runtimes with a memory
 * pool fixed in advance, embedders that only hand over tensors they own).
 * Same result as mla_latent_cache_append, same arguments minus the
 * workspace: the fp32 staging of the projection lives in a fixed 4 MiB
 * device array inside the library, held by every GPU that loads it until
 * the process exits.  Limits and rules:
 *  - n * (kv_lora_rank + qk_rope_head_dim) must fit 2^20 floats
 *    (mla_append_noalloc_max_tokens(h) tokens, 1820 at entry width 576);
 *    larger n returns MLA_ERR_INVALID_ARG with a message, nothing launched;
 *  - the handle's device must be current; the first call on each device
 *    looks up the array's device address (cudaGetSymbolAddress), so make
 *    that first call before any stream capture; the address is kept for the
 *    life of the process, so this entry point must not be used after the
 *    device has been reset (cudaDeviceReset destroys the array);
 *  - every call shares the one array per device: calls whose work overlaps
 *    on the GPU (other streams, other handles, other threads) race on it and
 *    must be ordered by the caller.  Nothing in it needs to start at zero.
 * Calls no cudaMalloc/cudaFree and no allocating library routine. */
mla_status_t mla_latent_cache_append_noalloc(mla_handle_t *h, const void *hidden,
                                             const int32_t *positions,
                                             const int64_t *slot_mapping, int32_t n,
                                             void *cache, int32_t num_pages, void *stream);
int64_t mla_append_noalloc_max_tokens(const mla_handle_t *h);

/* Byte offset inside a forward workspace (sized for num_tokens block tokens)
 * of an intermediate the forward leaves there: MLA_WS_Q_ABS, the absorbed
 * queries [num_tokens, H, kv_lora_rank + qk_rope_head_dim] in the cache dtype,
 * MLA_WS_O_LAT, the latent attention output [num_tokens, H, kv_lora_rank]
 * (fp16 for bf16 layers, fp32 for fp32 layers), or MLA_WS_O, the per-head
 * output [num_tokens, H, v_head_dim] that o_proj reads (same types; in a
 * workspace of mla_draft_forward_shared too, at the same offsets).  Valid after the forward's
 * work on the stream has completed, until the workspace is reused.  Returns
 * (size_t)-1 for a NULL handle, a negative count or an unknown part. */
size_t mla_forward_workspace_offset(const mla_handle_t *h, int32_t num_tokens,
                                    int32_t part);

/* The latent attention step alone (MLA blog, forward_mqa and the Triton
 * decode_attention_fwd it calls, which returns the output and the
 * log-sum-exp of each query row; PR #758 / PR #1026 masks and zeroing):
 * for every row m = (token, head) of q_abs,
 *   s_j = scale * <q_abs[m], cache entry of key j>   over the visible keys j
 *   o_lat[m] = sum_j softmax(s)_j * entry_j[:kv_lora_rank]
 *   lse[m]   = log sum_j exp(s_j)                     (natural log)
 * with visibility and the key -> cache-slot walk of mla_attn_desc_t.  A row
 * that sees no key gets o_lat = +0 exactly and lse = -inf.
 * q_abs: device [nb*T, H, kv_lora_rank + qk_rope_head_dim] in the cache dtype
 * (bf16 or fp32), 16-byte aligned; positions: device int32 [nb*T]; cache as
 * for the forward; o_lat: device [nb*T, H, kv_lora_rank], fp16 for bf16
 * layers (the forward's intermediate type), fp32 for fp32 layers; lse:
 * device fp32 [nb*T, H] or NULL.  The cache is only read.  Blocks of at
 * most 32 query rows (block_len * num_heads <= 32, bf16, page_size a
 * multiple of 128) run a kernel for few rows that splits every block's keys
 * across the SMs and merges the splits by log-sum-exp (the blog's
 * forward_mqa num_kv_splits / merge_attn_states); it needs a device
 * workspace of mla_latent_attention_workspace_bytes() (256-byte aligned;
 * MLA_ERR_INVALID_ARG when smaller), other shapes need none (workspace may be
 * NULL).  Asynchronous on `stream`; no allocation.  Index errors are
 * reported through the device status word like the forward's. */
size_t mla_latent_attention_workspace_bytes(const mla_handle_t *h, const mla_attn_desc_t *desc);
mla_status_t mla_latent_attention(mla_handle_t *h, const void *q_abs,
                                  const int32_t *positions, const void *cache,
                                  int32_t num_pages, const mla_attn_desc_t *desc,
                                  void *o_lat, float *lse, void *workspace,
                                  size_t workspace_bytes, void *stream);

/* Backward of the latent attention step (the draft layer is trained through
 * it: "Add config-selectable MLA draft attention" (SpecForge PR #758),
 * Validation, gradient parity; forward = mla_latent_attention).  With
 * P = exp(scale * <q_abs[i], e_j> - lse[i]) over the visible keys j of row
 * i, dP = d_o_lat[i] . e_j[:kv_lora_rank], D = d_o_lat[i] . o_lat[i] and
 * dS = P (dP - D):
 *   d_q_abs[i] = scale * sum_j dS_ij e_j                        (written)
 *   d_cache[slot(j)] += scale * sum_i dS_ij q_abs[i]
 *                       + sum_i P_ij d_o_lat[i] on its first kv_lora_rank
 *                         columns (the entries are keys and values at once)
 * over every block of `desc` (blocks whose keys share cache pages add into
 * the same slots; the caller zeroes d_cache before the first call).  Rows
 * without a visible key pass nothing back.  q_abs, positions, cache, desc as
 * for mla_latent_attention; o_lat and lse are that call's outputs; d_o_lat,
 * d_q_abs: device fp32 [nb*T, H, ...]; d_cache: device fp32 [num_pages *
 * page_size, kv_lora_rank + qk_rope_head_dim].  SIMT kernels, fp32
 * arithmetic; entries at most 640 wide (MLA_ERR_UNSUPPORTED otherwise).
 * Asynchronous on `stream`; no allocation. */
mla_status_t mla_latent_attention_backward(mla_handle_t *h, const void *q_abs,
                                           const int32_t *positions, const void *cache,
                                           int32_t num_pages, const mla_attn_desc_t *desc,
                                           const void *o_lat, const float *lse,
                                           const float *d_o_lat, float *d_q_abs,
                                           float *d_cache, void *stream);

/* Synchronise `stream`, read and clear the device status word.  Returns
 * MLA_OK, MLA_ERR_TIMEOUT (MLA_DEV_TIMEOUT set) or MLA_ERR_DEVICE_CHECK; the
 * raw bits go to *bits when non-NULL. */
mla_status_t mla_get_device_status(mla_handle_t *h, void *stream, int32_t *bits);

/* Self-check of the failure path (no counterpart on the pages: a test aid
 * for the bounded waits every kernel of the library uses).  Enqueues one
 * single-thread kernel that waits, with the library's bounded mbarrier wait,
 * on a barrier nothing ever arrives on; after max_rounds try_wait rounds
 * (1 .. 2^24; the kernels themselves use 2^26) the wait gives up, sets
 * MLA_DEV_TIMEOUT in the handle's device status word and writes 1 to
 * *gave_up (device int32).  The kernel issues no copies and holds no tensor
 * memory, so nothing is in flight when it returns and the handle stays
 * usable: mla_get_device_status then returns MLA_ERR_TIMEOUT once and clears
 * the word.  Asynchronous on `stream`. */
mla_status_t mla_check_wait_timeout(mla_handle_t *h, uint32_t max_rounds,
                                    int32_t *gave_up, void *stream);

/* Number of CUDA kernels this handle has enqueued so far (host counter;
 * launches replayed from a captured CUDA graph are not counted). */
unsigned long long mla_kernel_launches(const mla_handle_t *h);

void mla_draft_destroy(mla_handle_t *h);
const char *mla_status_string(mla_status_t s);
/* Message of the last failing call on this thread ("" if none). */
const char *mla_last_error(void);

#ifdef __cplusplus
}
#endif
#endif /* MLA_DRAFT_H */
