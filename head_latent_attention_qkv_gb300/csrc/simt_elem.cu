// Row-wise SIMT kernels: latent finish (RMSNorm + RoPE + cache store),
// query RMSNorm, query RoPE split (see simt.cuh).
#include "simt.cuh"

#include <math.h>

namespace mla {
namespace simt {

namespace {

constexpr int ROW_THREADS = 128;

// Sum of v over the CTA (blockDim.x == ROW_THREADS); every thread gets it.
__device__ float block_sum(float v) {
  __shared__ float part[ROW_THREADS / 32];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  const int w = threadIdx.x / 32;
  __syncthreads();
  if ((threadIdx.x & 31) == 0) part[w] = v;
  __syncthreads();
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < ROW_THREADS / 32; ++i) s += part[i];
  return s;
}

// Rotation pair k of a rope slice of width dr: element indices (ia, ib).
__device__ __forceinline__ void rope_pair(int k, int dr, int interleaved, int* ia, int* ib) {
  if (interleaved) { *ia = 2 * k; *ib = 2 * k + 1; }
  else { *ia = k; *ib = k + dr / 2; }
}

template <typename T>
__global__ void __launch_bounds__(ROW_THREADS)
kv_finish_kernel(const float* __restrict__ kv, long ld, const int32_t* __restrict__ positions,
                 const int64_t* __restrict__ slots, T* __restrict__ cache, long num_slots,
                 int rkv, int dr, float eps, const float* __restrict__ gamma,
                 const float2* __restrict__ rope, int max_pos, int interleaved,
                 uint32_t* status) {
  pdl_trigger();
  pdl_wait();
  const int t = blockIdx.x;
  const float* row = kv + (long)t * ld;
  const long slot = slots[t];
  const int p = positions[t];
  const bool bad_slot = slot < 0 || slot >= num_slots;
  const bool bad_pos = p < 0 || p >= max_pos;
  if (bad_slot || bad_pos) {
    if (threadIdx.x == 0)
      set_status(status, (bad_slot ? MLA_DEV_BAD_SLOT : 0) | (bad_pos ? MLA_DEV_BAD_POSITION : 0));
    return;
  }
  float ss = 0.f;
  for (int i = threadIdx.x; i < rkv; i += ROW_THREADS) ss = fmaf(row[i], row[i], ss);
  ss = block_sum(ss);
  const float rstd = 1.f / sqrtf(ss / (float)rkv + eps);
  T* dst = cache + slot * (long)(rkv + dr);
  for (int i = threadIdx.x; i < rkv; i += ROW_THREADS) dst[i] = from_f32<T>(row[i] * rstd * gamma[i]);
  const int half = dr / 2;
  for (int k = threadIdx.x; k < half; k += ROW_THREADS) {
    int ia, ib;
    rope_pair(k, dr, interleaved, &ia, &ib);
    const float2 cs = rope[(long)p * half + k];
    const float a = row[rkv + ia], b = row[rkv + ib];
    dst[rkv + ia] = from_f32<T>(a * cs.x - b * cs.y);
    dst[rkv + ib] = from_f32<T>(b * cs.x + a * cs.y);
  }
}

template <typename T>
__global__ void __launch_bounds__(ROW_THREADS)
rmsnorm_rows_kernel(const float* __restrict__ in, long ld, int n, const float* __restrict__ gamma,
                    float eps, T* __restrict__ out) {
  pdl_trigger();
  pdl_wait();
  const float* row = in + (long)blockIdx.x * ld;
  float ss = 0.f;
  for (int i = threadIdx.x; i < n; i += ROW_THREADS) ss = fmaf(row[i], row[i], ss);
  ss = block_sum(ss);
  const float rstd = 1.f / sqrtf(ss / (float)n + eps);
  T* o = out + (long)blockIdx.x * n;
  for (int i = threadIdx.x; i < n; i += ROW_THREADS) o[i] = from_f32<T>(row[i] * rstd * gamma[i]);
}

// One warp per (token, head): lanes copy q_nope and rotate the rope pairs
// (consecutive lanes touch consecutive elements).
template <typename TN, typename TQ>
__global__ void __launch_bounds__(ROW_THREADS)
q_rope_split_kernel(const float* __restrict__ q, long ldq, const int32_t* __restrict__ positions,
                    int M, int H, int dn, int dr, int rkv, const float2* __restrict__ rope,
                    int max_pos, int interleaved, uint32_t* status, TN* __restrict__ q_nope,
                    TQ* __restrict__ q_abs) {
  pdl_trigger();
  pdl_wait();
  const long w = (blockIdx.x * (long)ROW_THREADS + threadIdx.x) / 32;
  const int lane = threadIdx.x % 32;
  if (w >= (long)M * H) return;
  const int m = (int)(w / H), h = (int)(w % H);
  const int dqk = dn + dr, L = rkv + dr, half = dr / 2;
  const float* src = q + (long)m * ldq + (long)h * dqk;
  TN* nope = q_nope + w * dn;
  for (int d = lane; d < dn; d += 32) nope[d] = from_f32<TN>(src[d]);
  const int p = positions[m];
  const bool bad = p < 0 || p >= max_pos;
  if (bad && h == 0 && lane == 0) set_status(status, MLA_DEV_BAD_POSITION);
  TQ* dst = q_abs + w * L + rkv;
  for (int k = lane; k < half; k += 32) {
    int ia, ib;
    rope_pair(k, dr, interleaved, &ia, &ib);
    if (bad) {
      dst[ia] = from_f32<TQ>(0.f);
      dst[ib] = from_f32<TQ>(0.f);
      continue;
    }
    const float2 cs = rope[(long)p * half + k];
    const float a = src[dn + ia], b = src[dn + ib];
    dst[ia] = from_f32<TQ>(a * cs.x - b * cs.y);
    dst[ib] = from_f32<TQ>(b * cs.x + a * cs.y);
  }
}

}  // namespace

template <typename T>
void kv_finish(cudaStream_t st, const mla_handle* h, const float* kv, long ld, int n,
               const int32_t* positions, const int64_t* slots, T* cache, long num_slots, bool pdl) {
  if (n <= 0) return;
  const Layout& l = h->lay;
  Launch L(dim3(n), dim3(ROW_THREADS), 0, st, pdl);
  cudaLaunchKernelEx(&L.cfg, kv_finish_kernel<T>, kv, ld, positions, slots, cache, num_slots, l.rkv,
                     l.dr, (float)h->cfg.rms_norm_eps, h->gamma_kv, h->rope, h->cfg.max_position,
                     (int)(h->cfg.rope == MLA_ROPE_INTERLEAVED), h->status);
}

template <typename T>
void rmsnorm_rows(cudaStream_t st, const float* in, long ld, int M, int n, const float* gamma,
                  float eps, T* out, bool pdl) {
  if (M <= 0) return;
  Launch L(dim3(M), dim3(ROW_THREADS), 0, st, pdl);
  cudaLaunchKernelEx(&L.cfg, rmsnorm_rows_kernel<T>, in, ld, n, gamma, eps, out);
}

template <typename TN, typename TQ>
void q_rope_split(cudaStream_t st, const mla_handle* h, const float* q, long ldq, int M,
                  const int32_t* positions, TN* q_nope, TQ* q_abs, bool pdl) {
  if (M <= 0) return;
  const Layout& l = h->lay;
  const long warps = (long)M * l.H, per_block = ROW_THREADS / 32;
  Launch L(dim3((unsigned)((warps + per_block - 1) / per_block)), dim3(ROW_THREADS), 0, st, pdl);
  cudaLaunchKernelEx(&L.cfg, q_rope_split_kernel<TN, TQ>, q, ldq, positions, M, l.H, l.dn, l.dr,
                     l.rkv, h->rope, h->cfg.max_position, (int)(h->cfg.rope == MLA_ROPE_INTERLEAVED),
                     h->status, q_nope, q_abs);
}

#define MLA_INST(T)                                                                          \
  template void kv_finish<T>(cudaStream_t, const mla_handle*, const float*, long, int,      \
                             const int32_t*, const int64_t*, T*, long, bool);               \
  template void rmsnorm_rows<T>(cudaStream_t, const float*, long, int, int, const float*,   \
                                float, T*, bool);
MLA_INST(float)
MLA_INST(__nv_bfloat16)
MLA_INST(__half)
#undef MLA_INST
template void q_rope_split<float, float>(cudaStream_t, const mla_handle*, const float*, long, int,
                                         const int32_t*, float*, float*, bool);
template void q_rope_split<__half, __nv_bfloat16>(cudaStream_t, const mla_handle*, const float*,
                                                  long, int, const int32_t*, __half*,
                                                  __nv_bfloat16*, bool);

}  // namespace simt
}  // namespace mla
