// Merge of split-KV partial attention outputs ("MLA (Multi-Head Latent
// Attention)" blog, forward_mha: merge_attn_states combines two partial
// attentions by their log-sum-exp; forward_mqa: the KV range is split into
// num_kv_splits parts for parallelism).
//
// Split s of a row left o_s = (sum_j p_j c_j) / l_s (fp32, normalised over its
// own keys) and lse_s = m_s + log2(l_s) (exp2 domain; -inf when the split saw
// no visible key).  The merged row is sum_s w_s o_s / sum_s w_s with
// w_s = exp2(lse_s - max_s lse_s); a row no split saw stays exactly zero.
#include "attn_tc.cuh"

namespace mla {
namespace tc {
namespace {

constexpr int DV = 512;  // latent value width

__global__ void __launch_bounds__(256)
merge_kernel(const float* __restrict__ o_part, const float* __restrict__ lse_part, int splits,
             long rows, __half* __restrict__ o_lat, int32_t* vis_stats, int H) {
  pdl_trigger();
  pdl_wait();
  const long row = blockIdx.x * 8L + threadIdx.x / 32;   // one warp per row
  const int lane = threadIdx.x % 32;
  if (row >= rows) return;
  float mx = -INFINITY;
  for (int s = 0; s < splits; ++s) mx = fmaxf(mx, lse_part[s * rows + row]);
  float w[8], den = 0.f;
#pragma unroll
  for (int s = 0; s < 8; ++s) {
    w[s] = (s < splits && mx != -INFINITY) ? exp2f(lse_part[s * rows + row] - mx) : 0.f;
    den += w[s];
  }
  const float inv = den > 0.f ? 1.f / den : 0.f;
#pragma unroll
  for (int k = 0; k < DV / 32 / 4; ++k) {     // 4 float4 per lane
    const int c = (k * 32 + lane) * 4;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int s = 0; s < 8; ++s) {
      if (s < splits && w[s] > 0.f) {
        const float4 v = *reinterpret_cast<const float4*>(o_part + ((long)s * rows + row) * DV + c);
        acc.x += w[s] * v.x; acc.y += w[s] * v.y; acc.z += w[s] * v.z; acc.w += w[s] * v.w;
      }
    }
    __half2 h[2] = {__floats2half2_rn(acc.x * inv, acc.y * inv), __floats2half2_rn(acc.z * inv, acc.w * inv)};
    *reinterpret_cast<uint2*>(o_lat + row * DV + c) = *reinterpret_cast<uint2*>(h);
  }
  // visibility statistics were gathered with atomics: "no key" is first = INT_MAX
  if (vis_stats && lane == 0 && row % H == 0) {
    const long m = row / H;
    if (vis_stats[m * 3 + 1] == 0x7fffffff) vis_stats[m * 3 + 1] = -1;
  }
}

__global__ void vis_init_kernel(int32_t* vis_stats, long tokens) {
  pdl_trigger();
  pdl_wait();
  for (long i = blockIdx.x * (long)blockDim.x + threadIdx.x; i < tokens; i += (long)gridDim.x * blockDim.x) {
    vis_stats[i * 3 + 0] = 0;
    vis_stats[i * 3 + 1] = 0x7fffffff;
    vis_stats[i * 3 + 2] = -1;
  }
}

}  // namespace

void merge_splits(cudaStream_t st, const float* o_part, const float* lse_part, int splits,
                  long rows, __half* o_lat, int32_t* vis_stats, int H, bool pdl) {
  Launch L(dim3((unsigned)((rows + 7) / 8)), dim3(256), 0, st, pdl);
  cudaLaunchKernelEx(&L.cfg, merge_kernel, o_part, lse_part, splits, rows, o_lat, vis_stats, H);
}

void init_vis_stats(cudaStream_t st, int32_t* vis_stats, long tokens, bool pdl) {
  Launch L(dim3((unsigned)((tokens + 255) / 256 < 1024 ? (tokens + 255) / 256 : 1024)), dim3(256), 0,
           st, pdl);
  cudaLaunchKernelEx(&L.cfg, vis_init_kernel, vis_stats, tokens);
}

}  // namespace tc
}  // namespace mla
