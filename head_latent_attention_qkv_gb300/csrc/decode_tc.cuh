// tcgen05 latent attention for blocks of at most 32 query rows (see decode_tc.cu).
#pragma once

#include <cuda.h>

#include "common.cuh"

namespace mla {
namespace tc {

struct DecodeParams {
  CUtensorMap tmQ;    // Q_abs [rows, 576], chunked view, box 32 rows x 9 chunks
  CUtensorMap tmK1;   // cache [slots, 576], box 64 dims x 128 rows
  CUtensorMap tmK2;   // the same, chunked, box 128 rows x 2 chunks
  const int32_t* block_table;
  const int32_t* kv_len;
  const int32_t* window;
  const uint8_t* q_visible;
  const int32_t* positions;
  int32_t* vis_stats;
  __half* o_lat;      // [rows, 512]
  float* lse;         // [rows] or NULL
  float* part;        // [slots, 32, 512] normalised partial outputs, row major
  float* part_lse;    // [slots, 32] log2-sum-exp of each partial row
  int* part_vis;      // [slots, T, 3]
  int* meta;          // [blocks, 2]: first CTA, segment count
  uint32_t* status;
  int num_blocks, max_pages, num_pages, page_size, T, H;
  float scale_log2;
};

// True when the few-row kernel serves blocks of `block_len` tokens for this
// layer: bf16, kv_lora_rank 512, qk_rope 64, block_len * num_heads <= 32,
// page_size a multiple of 128.
bool decode_applies(const mla_handle* h, int block_len);
// Workspace of one launch (the segments' partial outputs, log-sum-exps,
// visibility counts and each block's segment range), 256-byte aligned pieces.
size_t decode_workspace_bytes(const mla_handle* h, const mla_attn_desc_t& desc);
// The same for any launch of at most max_blocks blocks of at most
// max_block_len tokens.
size_t decode_workspace_bound(const mla_handle* h, long max_blocks, int max_block_len);
// Latent attention of desc's blocks through the few-row kernel and the
// segment merge; same results as latent_attention() (o_lat, optional lse,
// vis_stats).  MLA_ERR_UNSUPPORTED when decode_applies() is false.
mla_status_t latent_decode(cudaStream_t st, const mla_handle* h, const __nv_bfloat16* q_abs,
                           const __nv_bfloat16* cache, int num_pages, const mla_attn_desc_t& desc,
                           const int32_t* positions, __half* o_lat, float* lse, void* workspace,
                           size_t workspace_bytes, bool pdl = false);

}  // namespace tc
}  // namespace mla
