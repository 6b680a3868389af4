// Backward of the latent attention step (the layer's training path: the
// draft attention is trained through this step, "Add config-selectable MLA
// draft attention" (SpecForge PR #758), Validation: gradient parity; the
// forward is the MLA blog's forward_mqa over the latent cache).
//
// For every query row i (a (token, head) pair of a block) and visible key j:
//   s_ij = scale <q_i, e_j>,  P_ij = exp(s_ij - lse_i)      (lse from the forward)
//   dP_ij = <dO_i, v_j>       (v_j = e_j[:kv_lora_rank])
//   D_i   = <dO_i, O_i>       (= sum_j P_ij dP_ij)
//   dS_ij = P_ij (dP_ij - D_i)
//   dQ_i  = scale sum_j dS_ij e_j
//   dE_j  = scale sum_i dS_ij q_i  +  sum_i P_ij dO_i  (the second term on the
//           first kv_lora_rank columns: the entries are keys and values at once)
// A row that sees no key has P = 0 and passes nothing back.
//
// SIMT, fp32 arithmetic.  dQ: one CTA per (block, head, 16 queries) loops over
// the block's keys in tiles of 32 staged in shared memory.  dE: one CTA per
// (block, 32 keys) loops over the block's rows 16 at a time and adds its
// keys' gradients into the caller's fp32 buffer with atomicAdd (blocks that
// share context pages add into the same slots).
#include "common.cuh"
#include "simt.cuh"

#include <math.h>

namespace mla {
namespace simt {
namespace {

constexpr int QT = 16, KT = 32, THREADS = 256, MAX_L = 640;

struct BwdArgs {
  const void* q_abs;          // [R, L] cache dtype
  const void* cache;          // [slots, L]
  const void* o_lat;          // [R, rkv] (fp16 for bf16 layers, fp32 for fp32)
  const float* lse;           // [R]
  const float* d_o;           // [R, rkv] fp32
  float* d_q;                 // [R, L] fp32 (written)
  float* d_cache;             // [slots, L] fp32 (added to)
  const int32_t* block_table; const int32_t* kv_len; const int32_t* window;
  const uint8_t* q_visible; const int32_t* positions;
  int num_pages, page_size, max_pages, T, H, rkv, L;
  float scale;
  uint32_t* status;
};

template <typename T> __device__ __forceinline__ float ld(const void* p, long i) {
  return to_f32(reinterpret_cast<const T*>(p)[i]);
}

// Effective key range of block b (kv_len clamped, a negative window rejected).
__device__ __forceinline__ int block_kvl(const BwdArgs& a, int b, int* W) {
  int kvl = a.kv_len[b];
  const int cap = a.max_pages * a.page_size;
  if (kvl < 0 || kvl > cap) {
    set_status(a.status, MLA_DEV_BAD_LENGTH);
    kvl = max(0, min(kvl, cap));
  }
  *W = a.window ? a.window[b] : 0;
  if (*W < 0) {
    set_status(a.status, MLA_DEV_BAD_WINDOW);
    kvl = 0;
  }
  return kvl;
}

// Cache slot of key j of block b, or -1 (invalid page: status set).
__device__ __forceinline__ long key_slot(const BwdArgs& a, int b, int j) {
  const int page = a.block_table[(long)b * a.max_pages + j / a.page_size];
  if (page < 0 || page >= a.num_pages) {
    set_status(a.status, MLA_DEV_BAD_PAGE);
    return -1;
  }
  return (long)page * a.page_size + j % a.page_size;
}

__device__ __forceinline__ bool visible(const BwdArgs& a, long m, int j, int kvl, int W) {
  const bool qv = a.q_visible ? a.q_visible[m] != 0 : true;
  return qv && j < kvl && (W == 0 || a.positions[m] - j < W);
}

// dQ: CTA (block b, head h, queries i0 .. i0+15); thread (r = tid / 16, c0 = tid % 16).
template <typename TC, typename TO>
__global__ void __launch_bounds__(THREADS) dq_kernel(const BwdArgs a) {
  extern __shared__ float sm[];
  const int L = a.L, rkv = a.rkv;
  float* Es = sm;                       // [KT][L + 1]
  float* Ps = Es + KT * (L + 1);        // [QT][KT] dS
  const int b = blockIdx.x, h = blockIdx.y, i0 = blockIdx.z * QT;
  const int nq = min(QT, a.T - i0);
  const int tid = threadIdx.x, r = tid / 16, c0 = tid % 16;
  const bool row_ok = r < nq;
  const long m = (long)b * a.T + i0 + r;          // token
  const long row = m * a.H + h;                   // Q_abs row
  int W;
  const int kvl = block_kvl(a, b, &W);
  // this row's lse and D = <dO, O> (16 threads of the row, shuffled)
  const float lse = row_ok ? a.lse[row] : -INFINITY;
  float D = 0.f;
  if (row_ok)
    for (int d = c0; d < rkv; d += 16) D += a.d_o[row * rkv + d] * ld<TO>(a.o_lat, row * rkv + d);
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) D += __shfl_xor_sync(0xffffffffu, D, o);
  const int nout = (L + 15) / 16;
  float acc[MAX_L / 16];
#pragma unroll
  for (int i = 0; i < MAX_L / 16; ++i) acc[i] = 0.f;
  for (int j0 = 0; j0 < kvl; j0 += KT) {
    __syncthreads();
    for (int idx = tid; idx < KT * L; idx += THREADS) {
      const int kk = idx / L, d = idx % L, j = j0 + kk;
      float v = 0.f;
      if (j < kvl) {
        const long sl = key_slot(a, b, j);
        if (sl >= 0) v = ld<TC>(a.cache, sl * L + d);
      }
      Es[kk * (L + 1) + d] = v;
    }
    __syncthreads();
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int kk = c0 + 16 * u, j = j0 + kk;
      float ds = 0.f;
      if (row_ok && lse != -INFINITY && visible(a, m, j, kvl, W)) {
        const float* e = Es + kk * (L + 1);
        float s = 0.f, dp = 0.f;
        for (int d = 0; d < L; ++d) s = fmaf(ld<TC>(a.q_abs, row * L + d), e[d], s);
        for (int d = 0; d < rkv; ++d) dp = fmaf(a.d_o[row * rkv + d], e[d], dp);
        const float p = expf(s * a.scale - lse);
        ds = p * (dp - D);
      }
      Ps[r * KT + kk] = ds;
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < MAX_L / 16; ++i) {
      const int d = c0 + 16 * i;
      if (i < nout && d < L) {
        float s = acc[i];
        for (int k = 0; k < KT; ++k) s = fmaf(Ps[r * KT + k], Es[k * (L + 1) + d], s);
        acc[i] = s;
      }
    }
  }
  if (row_ok) {
#pragma unroll
    for (int i = 0; i < MAX_L / 16; ++i) {
      const int d = c0 + 16 * i;
      if (i < nout && d < L) a.d_q[row * L + d] = a.scale * acc[i];
    }
  }
}

// dE: CTA (block b, keys j0 .. j0+31); thread (k = tid / 8 key, part = tid % 8
// of its dims).  Rows of the block are visited 16 at a time.
template <typename TC, typename TO>
__global__ void __launch_bounds__(THREADS) de_kernel(const BwdArgs a) {
  extern __shared__ float sm[];
  const int L = a.L, rkv = a.rkv;
  float* Qs = sm;                       // [QT][L]
  float* Os = Qs + QT * L;              // [QT][rkv] dO
  float* Gs = Os + QT * rkv;            // [QT][KT] dS (scaled), then P
  float* Ps = Gs + QT * KT;             // [QT][KT] P
  float* Ds = Ps + QT * KT;             // [QT] D
  float* Ls = Ds + QT;                  // [QT] lse
  const int b = blockIdx.x, j0 = blockIdx.y * KT;
  int W;
  const int kvl = block_kvl(a, b, &W);
  if (j0 >= kvl) return;
  const int tid = threadIdx.x, k = tid / 8, part = tid % 8;
  const int j = j0 + k;
  const bool key_ok = j < kvl;
  const long sl = key_ok ? key_slot(a, b, j) : -1;
  // this thread's share of the key's entry: dims part, part + 8, ...
  const int nd = (L + 7) / 8;
  float e[MAX_L / 8], g[MAX_L / 8];
#pragma unroll
  for (int i = 0; i < MAX_L / 8; ++i) {
    const int d = part + 8 * i;
    e[i] = (i < nd && d < L && sl >= 0) ? ld<TC>(a.cache, sl * L + d) : 0.f;
    g[i] = 0.f;
  }
  const long rows = (long)a.T * a.H;
  for (long r0 = 0; r0 < rows; r0 += QT) {
    const int nr = (int)min((long)QT, rows - r0);
    __syncthreads();
    for (int idx = tid; idx < QT * L; idx += THREADS) {
      const int rr = idx / L, d = idx % L;
      Qs[idx] = rr < nr ? ld<TC>(a.q_abs, ((long)b * rows + r0 + rr) * L + d) : 0.f;
    }
    for (int idx = tid; idx < QT * rkv; idx += THREADS) {
      const int rr = idx / rkv, d = idx % rkv;
      Os[idx] = rr < nr ? a.d_o[((long)b * rows + r0 + rr) * rkv + d] : 0.f;
    }
    if (tid < QT) {
      const long row = (long)b * rows + r0 + tid;
      float D = 0.f;
      if (tid < nr)
        for (int d = 0; d < rkv; ++d) D += a.d_o[row * rkv + d] * ld<TO>(a.o_lat, row * rkv + d);
      Ds[tid] = D;
      Ls[tid] = tid < nr ? a.lse[row] : -INFINITY;
    }
    __syncthreads();
    // s, dP for (row rr, key k): the 8 threads of key k split the dims
    for (int rr = 0; rr < QT; ++rr) {
      float s = 0.f, dp = 0.f;
#pragma unroll
      for (int i = 0; i < MAX_L / 8; ++i) {
        const int d = part + 8 * i;
        if (i < nd && d < L) {
          s = fmaf(Qs[rr * L + d], e[i], s);
          if (d < rkv) dp = fmaf(Os[rr * rkv + d], e[i], dp);
        }
      }
#pragma unroll
      for (int o = 4; o > 0; o >>= 1) {
        s += __shfl_xor_sync(0xffffffffu, s, o);
        dp += __shfl_xor_sync(0xffffffffu, dp, o);
      }
      const long row = (long)b * rows + r0 + rr;
      const long m = row / a.H;
      const bool vis = rr < nr && key_ok && sl >= 0 && Ls[rr] != -INFINITY && visible(a, m, j, kvl, W);
      const float p = vis ? expf(s * a.scale - Ls[rr]) : 0.f;
      if (part == 0) {
        Gs[rr * KT + k] = a.scale * p * (dp - Ds[rr]);
        Ps[rr * KT + k] = p;
      }
    }
    __syncwarp();
    // accumulate: g[d] += sum_rr dS * q[rr][d] + P * dO[rr][d] (d < rkv)
    for (int rr = 0; rr < QT; ++rr) {
      const float ds = Gs[rr * KT + k], p = Ps[rr * KT + k];
#pragma unroll
      for (int i = 0; i < MAX_L / 8; ++i) {
        const int d = part + 8 * i;
        if (i < nd && d < L) {
          float v = fmaf(ds, Qs[rr * L + d], g[i]);
          if (d < rkv) v = fmaf(p, Os[rr * rkv + d], v);
          g[i] = v;
        }
      }
    }
  }
  if (sl >= 0) {
#pragma unroll
    for (int i = 0; i < MAX_L / 8; ++i) {
      const int d = part + 8 * i;
      if (i < nd && d < L) atomicAdd(a.d_cache + sl * L + d, g[i]);
    }
  }
}

template <typename TC, typename TO>
void launch(cudaStream_t st, const BwdArgs& a, int num_blocks, int max_kv) {
  const size_t sm_dq = sizeof(float) * (KT * (a.L + 1) + QT * KT);
  const size_t sm_de = sizeof(float) * (QT * a.L + QT * a.rkv + 2 * QT * KT + 2 * QT);
  static bool configured = false;
  if (!configured) {
    cudaFuncSetAttribute(dq_kernel<TC, TO>, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
    cudaFuncSetAttribute(de_kernel<TC, TO>, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
    configured = true;
  }
  dq_kernel<TC, TO><<<dim3(num_blocks, a.H, (a.T + QT - 1) / QT), THREADS, sm_dq, st>>>(a);
  de_kernel<TC, TO><<<dim3(num_blocks, (max_kv + KT - 1) / KT), THREADS, sm_de, st>>>(a);
}

}  // namespace
}  // namespace simt
}  // namespace mla

extern "C" mla_status_t mla_latent_attention_backward(
    mla_handle_t* h, const void* q_abs, const int32_t* positions, const void* cache,
    int32_t num_pages, const mla_attn_desc_t* desc, const void* o_lat, const float* lse,
    const float* d_o_lat, float* d_q_abs, float* d_cache, void* stream) {
  using namespace mla;
  if (!h || !desc) return fail(MLA_ERR_INVALID_ARG, "attention backward: null handle or descriptor");
  const mla_attn_desc_t& d = *desc;
  if (d.num_blocks < 0 || d.block_len <= 0 || d.max_pages <= 0)
    return fail(MLA_ERR_INVALID_ARG, "attention backward: num_blocks >= 0, block_len > 0, max_pages > 0");
  if (d.num_blocks == 0) return MLA_OK;
  if (!q_abs || !positions || !cache || !o_lat || !lse || !d_o_lat || !d_q_abs || !d_cache ||
      !d.block_table || !d.kv_len)
    return fail(MLA_ERR_INVALID_ARG, "attention backward: null pointer");
  if (num_pages <= 0) return fail(MLA_ERR_INVALID_ARG, "attention backward: num_pages <= 0");
  const Layout& l = h->lay;
  if (l.L > simt::MAX_L) return fail(MLA_ERR_UNSUPPORTED, "attention backward: entry wider than 640");
  const int max_kv = d.max_pages * h->cfg.page_size;
  simt::BwdArgs a{q_abs, cache, o_lat, lse, d_o_lat, d_q_abs, d_cache, d.block_table, d.kv_len,
                  d.window, d.q_visible, positions, num_pages, h->cfg.page_size, d.max_pages,
                  d.block_len, l.H, l.rkv, l.L, h->scale, h->status};
  cudaStream_t st = (cudaStream_t)stream;
  h->launches += 2;
  if (h->cfg.dtype == MLA_BF16)
    simt::launch<__nv_bfloat16, __half>(st, a, d.num_blocks, max_kv);
  else
    simt::launch<float, float>(st, a, d.num_blocks, max_kv);
  MLA_CUDA_TRY(cudaGetLastError());
  return MLA_OK;
}
