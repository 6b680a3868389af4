// SIMT (CUDA-core, fp32-accumulate) kernels of the MLA draft layer.
// `pdl`: launch with programmatic stream serialization (the kernel waits for
// the previous kernel of the stream with griddepcontrol.wait).
//
// These are the production path for the fp32 configuration (tensor-core
// TF32 would not meet a 1e-4 relative tolerance) and the first, plain
// implementation of every step for bf16.  Storage types: fp32 throughout for
// the fp32 configuration; for bf16 layers the hidden states, A-projection
// weights and latent cache are bf16 while the intermediate activations
// (normed q_c, q_nope, Q_abs, O_lat, o) and the weights they meet are fp16,
// whose 3 extra mantissa bits keep the rounding of these tensor-core operands
// well inside the output tolerance.  Every sum is accumulated in fp32.
#pragma once

#include "common.cuh"

namespace mla {
namespace simt {

// C[z][m][n] = sum_k A[z][m][k] * B[z][n][k]  (both operands K-contiguous, the
// torch.nn.Linear product x @ W^T), optionally multiplied by sigmoid(G[z][m][n])
// (G fp32).  Leading dims / batch strides are in elements.
template <typename TA, typename TC>
void gemm_nt(cudaStream_t st, int M, int N, int K, int batch,
             const TA* A, long lda, long sA, const TA* B, long ldb, long sB,
             TC* C, long ldc, long sC, const float* G, long ldg, long sG);

// Latent entry of each of n tokens from its raw kv row (fp32, row stride ld):
// cache[slot] = [RMSNorm(kv[:rkv]) * gamma | RoPE(kv[rkv:], pos)].
template <typename T>
void kv_finish(cudaStream_t st, const mla_handle* h, const float* kv, long ld, int n,
               const int32_t* positions, const int64_t* slots, T* cache, long num_slots,
               bool pdl = false);

// out[m][:] = RMSNorm(in[m][:n]) * gamma  (in fp32 with row stride ld).
template <typename T>
void rmsnorm_rows(cudaStream_t st, const float* in, long ld, int M, int n,
                  const float* gamma, float eps, T* out, bool pdl = false);

// q [M, H, dqk] fp32 (row stride ldq) -> q_nope [M, H, dn] and the rotated
// rope part into Q_abs[m, h, rkv:rkv+dr].
template <typename TN, typename TQ>
void q_rope_split(cudaStream_t st, const mla_handle* h, const float* q, long ldq, int M,
                  const int32_t* positions, TN* q_nope, TQ* q_abs, bool pdl = false);

// Latent attention: O_lat[m, h, :rkv] = sum_j p_j c_j over the visible keys of
// each query's block, scores scale * <Q_abs[m,h,:], entry_j>; optionally the
// rows' log-sum-exp of the scaled scores (lse[m * H + h], -inf without keys).
template <typename TQ, typename TC>
void latent_attention(cudaStream_t st, const mla_handle* h, const TQ* q_abs,
                      const TC* cache, int num_pages, const mla_attn_desc_t& desc,
                      const int32_t* positions, TQ* o_lat, float* lse = nullptr);

}  // namespace simt
}  // namespace mla
