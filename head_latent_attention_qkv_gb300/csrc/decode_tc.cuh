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
  CUtensorMap tmK4;   // the same, chunked, box 128 rows x 4 chunks
  const int32_t* block_table;
  const int32_t* kv_len;
  const int32_t* window;
  const uint8_t* q_visible;
  const int32_t* positions;
  int32_t* vis_stats;
  __half* o_lat;      // [rows, 512]
  float* lse;         // [rows] or NULL
  float* part;        // [blocks, splits, 32, 512] normalised partial outputs
  float* part_lse;    // [blocks, splits, 32] log2-sum-exp of each partial
  int* part_vis;      // [blocks, splits, T, 3]
  uint32_t* status;
  int max_pages, num_pages, page_size, T, H, splits, tiles_per_split;
  float scale_log2;
};

// True when the few-row kernel serves blocks of `block_len` tokens for this
// layer: bf16, kv_lora_rank 512, qk_rope 64, block_len * num_heads <= 32,
// page_size a multiple of 128.
bool decode_applies(const mla_handle* h, int block_len);
// Workspace of one launch (the splits' partial outputs, log-sum-exps and
// visibility counts), 256-byte aligned pieces.
size_t decode_workspace_bytes(const mla_handle* h, const mla_attn_desc_t& desc);
// Latent attention of desc's blocks through the few-row kernel and the
// split merge; same results as latent_attention() (o_lat, optional lse,
// vis_stats).  MLA_ERR_UNSUPPORTED when decode_applies() is false.
mla_status_t latent_decode(cudaStream_t st, const mla_handle* h, const __nv_bfloat16* q_abs,
                           const __nv_bfloat16* cache, int num_pages, const mla_attn_desc_t& desc,
                           const int32_t* positions, __half* o_lat, float* lse, void* workspace,
                           size_t workspace_bytes, bool pdl = false);

}  // namespace tc
}  // namespace mla
