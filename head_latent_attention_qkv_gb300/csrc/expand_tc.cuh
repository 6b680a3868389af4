// Expanded-form attention for blocks that share a context (see expand_tc.cu).
#pragma once

#include <cuda.h>

#include "common.cuh"

namespace mla {
namespace tc {

// Rows of the gathered latent buffer: every context's keys (ctx.ctx_rows),
// then every block's own keys (block_len per block).
inline long expand_rows(const mla_shared_ctx_t& ctx, int num_blocks, int block_len) {
  return (long)ctx.ctx_rows + (long)num_blocks * block_len;
}

// True when the expanded attention takes each context's blocks in units of
// one mask class (block_len a multiple of 8 dividing 128: the condition
// expanded_attention tests), which costs one more kernel, the pre-pass
// that orders the blocks.
inline bool expand_grouped(int block_len) { return block_len % 8 == 0 && 128 % block_len == 0; }

// True when the expanded attention serves these blocks: bf16 layer,
// kv_lora_rank 512, qk_rope 64, qk_nope 128, v_head 128, block_len <= 128.
bool expand_applies(const mla_handle* h, int block_len);

// Gathers the cache entries of each context (keys 0 .. ctx_len - 1 of the
// context's first block) and of each block's own keys (keys ctx_len ..
// ctx_len + block_len - 1 of the block) into dense bf16 rows
// out[expand_rows, 576] (a page outside the cache: zeros, MLA_DEV_BAD_PAGE).
void expand_gather(cudaStream_t st, const mla_handle* h, const __nv_bfloat16* cache, int num_pages,
                   const mla_attn_desc_t& d, const mla_shared_ctx_t& ctx, __nv_bfloat16* out, bool pdl);

// Every block's queries over its context's keys and its own keys in the
// expanded form: scores q_nope[h] . k_nope[h] + q_pe[h] . k_pe, o[h] =
// softmax . v[h] (times the gate when non-NULL).  q_nope fp16 [M, H, 128];
// q_abs bf16 [M, H, 576] (q_pe in dims 512..575); kv fp16 [rows, H, 256]
// (k_nope | v of each head: the gathered rows times kv_b_proj^T); gathered
// bf16 [rows, 576] (k_pe in dims 512..575); gate fp32 (row m, head h, dim d
// at gate[m * ld_gate + h * 128 + d]) or NULL; o fp16 [M, H, 128];
// unit_ws: device scratch of num_blocks + 2 * num_ctx int32 (the block order
// of the units).
mla_status_t expanded_attention(cudaStream_t st, const mla_handle* h, const __half* q_nope,
                                const __nv_bfloat16* q_abs, const __half* kv,
                                const __nv_bfloat16* gathered, long rows, const mla_attn_desc_t& d,
                                const mla_shared_ctx_t& ctx, const int32_t* positions,
                                const float* gate, long ld_gate, __half* o, int32_t* unit_ws, bool pdl);

}  // namespace tc
}  // namespace mla
