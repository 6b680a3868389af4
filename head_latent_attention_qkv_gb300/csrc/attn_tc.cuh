// tcgen05 latent attention launcher (see attn_tc.cu).
#pragma once

#include <cuda.h>

#include "common.cuh"

namespace mla {
namespace tc {

struct AttnParams {
  CUtensorMap tmQ;    // Q_abs bf16 [rows, 576], box 64 x 128
  CUtensorMap tmKV;   // latent cache bf16 [num_pages * page_size, 576], box 64 x seg_rows
  const int32_t* block_table;
  const int32_t* kv_len;
  const int32_t* window;
  const uint8_t* q_visible;
  const int32_t* positions;
  int32_t* vis_stats;
  __half* o_lat;      // [rows, 512]
  uint32_t* status;
  int max_pages, num_pages, page_size, seg_rows, T, H, tiles_per_block;
  float scale_log2;   // softmax scale * log2(e)
};

// Supported: kv_lora_rank 512, qk_rope 64, block_len * num_heads a multiple
// of 128, page_size a multiple of 16 (or of 64).  Returns
// MLA_ERR_UNSUPPORTED otherwise.
mla_status_t latent_attention(cudaStream_t st, const mla_handle* h, const __nv_bfloat16* q_abs,
                              const __nv_bfloat16* cache, int num_pages,
                              const mla_attn_desc_t& desc, const int32_t* positions,
                              __half* o_lat);

}  // namespace tc
}  // namespace mla
