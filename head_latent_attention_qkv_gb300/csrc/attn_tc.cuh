// tcgen05 latent attention launcher (see attn_tc.cu).
#pragma once

#include <cuda.h>

#include "common.cuh"

namespace mla {
namespace tc {

struct AttnParams {
  CUtensorMap tmQ;    // Q_abs bf16 [rows, 576], chunked view, box 128 rows x 7 chunks
  CUtensorMap tmK;    // latent cache bf16 [num_pages * page_size, 576], box 64 x 128 rows
  CUtensorMap tmKs;   // the same, box 64 x seg_rows (one page or 128 rows)
  CUtensorMap tmV;    // the cache, chunked view, box 128 rows x 4 chunks
  const __nv_bfloat16* q_abs;   // the same Q_abs (dims 0..127 go to tensor memory)
  const int32_t* block_table;
  const int32_t* kv_len;
  const int32_t* window;
  const uint8_t* q_visible;
  const int32_t* positions;
  int32_t* vis_stats;
  __half* o_lat;      // [rows, 512]
  float* lse;         // [rows] natural-log sum of exp of the scaled scores, or NULL
  int splits;         // key-range parts of a unit (1..4; cluster of 2 x splits CTAs)
  uint32_t* status;
  int max_pages, num_pages, page_size, seg_rows, T, H, tiles_per_block;
  float scale_log2;   // softmax scale * log2(e)
};

// Supported: kv_lora_rank 512, qk_rope 64, page_size 16, 32, 64 or a multiple
// of 128 (any block_len: a block's block_len * num_heads rows are processed in
// tiles of 128, the last one padded).  Returns MLA_ERR_UNSUPPORTED otherwise.
// The key range of every (block, 128-row) unit is split in attn_splits()
// parts when units alone do not fill the GPU; the parts are merged by
// log-sum-exp inside the kernel (no workspace).
int attn_splits(const mla_handle* h, long num_blocks, int block_len);
// `pdl`: the kernels may start while the previous kernel of the stream
// finishes (programmatic stream serialization; they wait for it on the device).
// `lse` (nullable): per Q_abs row, log of the sum over visible keys of
// exp(scale * score), -inf for a row that sees no key.
mla_status_t latent_attention(cudaStream_t st, const mla_handle* h, const __nv_bfloat16* q_abs,
                              const __nv_bfloat16* cache, int num_pages,
                              const mla_attn_desc_t& desc, const int32_t* positions,
                              __half* o_lat, float* lse = nullptr, bool pdl = false);

}  // namespace tc
}  // namespace mla
