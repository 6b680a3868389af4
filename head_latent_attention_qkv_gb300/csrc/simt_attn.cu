// SIMT latent attention (see simt.cuh).  One CTA per (block, head, chunk of
// up to 16 queries); key tiles of 32 cache entries are staged in shared memory
// as fp32 and an online softmax (fp32) runs over them.  Used for the fp32
// configuration.
#include "simt.cuh"

#include <math.h>

namespace mla {
namespace simt {

namespace {

constexpr int QT = 16, KT = 32, A_THREADS = 256, MAX_OUT = 32;  // rkv <= 16 * MAX_OUT

__device__ __forceinline__ float hmax16(float v) {
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float hsum16(float v) {
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ int hmaxi16(int v) {
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ int hsumi16(int v) {
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

template <typename TQ, typename TC>
__global__ void __launch_bounds__(A_THREADS)
latent_attn_kernel(const TQ* __restrict__ q_abs, const TC* __restrict__ cache, int num_pages,
                   int page_size, const int32_t* __restrict__ block_table, int max_pages,
                   const int32_t* __restrict__ kv_len, const int32_t* __restrict__ window,
                   const uint8_t* __restrict__ q_visible, const int32_t* __restrict__ positions,
                   int Tb, int H, int rkv, int L, float scale, uint32_t* status,
                   int32_t* vis_stats, TQ* __restrict__ o_lat, float* __restrict__ lse) {
  extern __shared__ float sm[];
  float* Qs = sm;                      // [QT][L]
  float* Ks = Qs + QT * L;             // [KT][L + 1]
  float* Ps = Ks + KT * (L + 1);       // [QT][KT]
  const int b = blockIdx.x, h = blockIdx.y, i0 = blockIdx.z * QT;
  const int nq = min(QT, Tb - i0);
  const int tid = threadIdx.x, r = tid / 16, c0 = tid % 16;
  const bool row_ok = r < nq;
  const long m = (long)b * Tb + i0 + r;
  const int p = row_ok ? positions[m] : 0;
  const bool qv = row_ok && (q_visible ? q_visible[m] != 0 : true);
  int kvl = kv_len[b];
  if (kvl < 0 || kvl > max_pages * page_size) {
    if (tid == 0) set_status(status, MLA_DEV_BAD_LENGTH);
    kvl = max(0, min(kvl, max_pages * page_size));
  }
  const int W = window ? window[b] : 0;
  if (W < 0) {                 // rejected: the block's rows see no key (exact zeros)
    if (tid == 0 && h == 0 && blockIdx.z == 0) set_status(status, MLA_DEV_BAD_WINDOW);
    kvl = 0;
  }
  // first key any query of this chunk can see
  int j_lo = 0;
  if (W > 0) {
    int pmin = 0x7fffffff;
    for (int i = 0; i < nq; ++i) pmin = min(pmin, positions[(long)b * Tb + i0 + i]);
    j_lo = max(0, pmin - W + 1);
  }
  for (int idx = tid; idx < QT * L; idx += A_THREADS) {
    const int rr = idx / L, d = idx % L;
    Qs[idx] = rr < nq ? to_f32(q_abs[(((long)b * Tb + i0 + rr) * H + h) * L + d]) : 0.f;
  }
  const int nout = rkv / 16;
  float o[MAX_OUT];
#pragma unroll
  for (int i = 0; i < MAX_OUT; ++i) o[i] = 0.f;
  float mrow = -INFINITY, lrow = 0.f;
  int cnt = 0, last = -1, first = 0x7fffffff;
  for (int j0 = j_lo; j0 < kvl; j0 += KT) {
    __syncthreads();
    for (int idx = tid; idx < KT * L; idx += A_THREADS) {
      const int kk = idx / L, d = idx % L, j = j0 + kk;
      float v = 0.f;
      if (j < kvl) {
        const int page = block_table[(long)b * max_pages + j / page_size];
        if (page >= 0 && page < num_pages)
          v = to_f32(cache[((long)page * page_size + j % page_size) * L + d]);
        else if (d == 0)
          set_status(status, MLA_DEV_BAD_PAGE);
      }
      Ks[kk * (L + 1) + d] = v;
    }
    __syncthreads();
    float s[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int kk = c0 + 16 * u, j = j0 + kk;
      const bool vis = qv && j < kvl && (W == 0 || p - j < W);
      s[u] = -INFINITY;
      if (vis) {
        float acc = 0.f;
        const float* qr = Qs + r * L;
        const float* kr = Ks + kk * (L + 1);
        for (int d = 0; d < L; ++d) acc = fmaf(qr[d], kr[d], acc);
        s[u] = acc * scale;
        ++cnt;
        first = min(first, j);
        last = max(last, j);
      }
    }
    const float m_new = fmaxf(mrow, hmax16(fmaxf(s[0], s[1])));
    const float alpha = (mrow == -INFINITY) ? 0.f : expf(mrow - m_new);
    const float p0 = (s[0] == -INFINITY) ? 0.f : expf(s[0] - m_new);
    const float p1 = (s[1] == -INFINITY) ? 0.f : expf(s[1] - m_new);
    lrow = lrow * alpha + hsum16(p0 + p1);
    mrow = m_new;
    Ps[r * KT + c0] = p0;
    Ps[r * KT + c0 + 16] = p1;
    __syncthreads();
#pragma unroll
    for (int i = 0; i < MAX_OUT; ++i) {
      if (i < nout) {
        const int c = c0 + 16 * i;
        float acc = o[i] * alpha;
        for (int k = 0; k < KT; ++k) acc = fmaf(Ps[r * KT + k], Ks[k * (L + 1) + c], acc);
        o[i] = acc;
      }
    }
  }
  if (row_ok) {
    const float inv = lrow > 0.f ? 1.f / lrow : 0.f;
    TQ* dst = o_lat + (m * H + h) * rkv;
#pragma unroll
    for (int i = 0; i < MAX_OUT; ++i)
      if (i < nout) dst[c0 + 16 * i] = from_f32<TQ>(lrow > 0.f ? o[i] * inv : 0.f);
    if (lse && c0 == 0) lse[m * H + h] = lrow > 0.f ? mrow + logf(lrow) : -INFINITY;
  }
  const int tot = hsumi16(cnt), hi = hmaxi16(last), lo = -hmaxi16(-first);
  if (vis_stats && h == 0 && row_ok && c0 == 0) {
    vis_stats[m * 3 + 0] = tot;
    vis_stats[m * 3 + 1] = tot ? lo : -1;
    vis_stats[m * 3 + 2] = tot ? hi : -1;
  }
}

}  // namespace

template <typename TQ, typename TC>
void latent_attention(cudaStream_t st, const mla_handle* h, const TQ* q_abs, const TC* cache,
                      int num_pages, const mla_attn_desc_t& desc, const int32_t* positions,
                      TQ* o_lat, float* lse) {
  const Layout& l = h->lay;
  if (desc.num_blocks <= 0 || desc.block_len <= 0) return;
  const size_t smem = sizeof(float) * (QT * l.L + KT * (l.L + 1) + QT * KT);
  static bool configured = false;
  if (!configured) {
    cudaFuncSetAttribute(latent_attn_kernel<TQ, TC>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         227 * 1024);
    configured = true;
  }
  dim3 grid(desc.num_blocks, l.H, (desc.block_len + QT - 1) / QT);
  latent_attn_kernel<TQ, TC><<<grid, A_THREADS, smem, st>>>(
      q_abs, cache, num_pages, h->cfg.page_size, desc.block_table, desc.max_pages, desc.kv_len,
      desc.window, desc.q_visible, positions, desc.block_len, l.H, l.rkv, l.L, h->scale,
      h->status, desc.vis_stats, o_lat, lse);
}

template void latent_attention<float, float>(cudaStream_t, const mla_handle*, const float*,
                                             const float*, int, const mla_attn_desc_t&,
                                             const int32_t*, float*, float*);
}  // namespace simt
}  // namespace mla
