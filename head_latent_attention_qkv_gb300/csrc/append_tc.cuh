// tcgen05 latent-cache append (see append_tc.cu).
#pragma once

#include "common.cuh"

namespace mla {
namespace tc {

// cache[slots[t]] = [RMSNorm(hidden[t] @ W_kva^T [:512]) * gamma | RoPE(... [512:], positions[t])]
// for t < M, bf16, one kernel (no workspace).  Needs kv_lora_rank 512 and
// qk_rope_head_dim 64 (MLA_ERR_UNSUPPORTED otherwise).
// `pdl`: may start while the previous kernel of the stream finishes.
mla_status_t kv_append(cudaStream_t st, const mla_handle* h, const __nv_bfloat16* hidden, int M,
                       const int32_t* positions, const int64_t* slots, __nv_bfloat16* cache,
                       long num_slots, bool pdl = false);

}  // namespace tc
}  // namespace mla
