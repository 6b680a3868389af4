// Latent-cache append on tcgen05 ("MLA (Multi-Head Latent Attention)" blog,
// wrapper forward + do_kv_cache_update / concat_and_cache_mla):
//   kv = hidden @ W_kva^T                     (W_kva: the kv_lora_rank + qk_rope rows)
//   cache[slot] = [RMSNorm(kv[:512]) * gamma | RoPE(kv[512:], position)]   (bf16)
//
// A cluster of three CTAs owns 128 token rows; CTA c computes output columns
// [192c, 192c + 192) in tensor memory.  CTA 0 multicasts each 128 x 64 slice of
// the hidden states to all three (each cluster reads the hidden rows once),
// each CTA streams its own 192 weight rows.  In the epilogue every CTA adds the
// squares of its latent columns per row, the three partial sums are exchanged
// through distributed shared memory and added in the same order everywhere,
// and each CTA normalises, rotates (CTA 2 holds the 64 rope columns) and
// stores its part of every row straight to the row's cache slot.
#include "append_tc.cuh"

#include <mutex>

#include "gemm_tc.cuh"
#include "tc_ptx.cuh"

namespace mla {
namespace tc {
namespace {

constexpr int BM = 128, BN = 192, BK = 64, THREADS = 128, STAGES = 5, CL = 3;
constexpr int A_BYTES = BM * BK * 2, B_BYTES = BN * BK * 2, STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int OFF_BAR = STAGES * STAGE_BYTES;
constexpr int SMEM_BYTES = 1024 + OFF_BAR + 1024;
constexpr uint32_t TMEM_COLS = 256;

struct AppendParams {
  CUtensorMap tmA;            // hidden [M, D]
  CUtensorMap tmB;            // W_kva [576, D]
  int M, K;
  const int32_t* positions;
  const int64_t* slots;
  __nv_bfloat16* cache;       // [num_slots, 576]
  long num_slots;
  const float* gamma;         // kv_a_layernorm, fp32 [512]
  const float2* rope;         // [max_pos, 32] (cos, sin)
  int max_pos, interleaved;
  float eps;
  uint32_t* status;
};

__global__ void __launch_bounds__(THREADS, 1) kv_append_tc_kernel(const __grid_constant__ AppendParams P) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint64_t* full = (uint64_t*)(smem + OFF_BAR);
  uint64_t* empty = full + STAGES;
  uint64_t* accum = empty + STAGES;
  uint32_t* tmem_slot = (uint32_t*)(accum + 1);
  float* red = (float*)(smem + OFF_BAR + 256);     // per-row partial sum of squares [128]

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const uint32_t rank = cluster_ctarank();         // == blockIdx.x: column block
  const int m0 = blockIdx.y * BM, n0 = (int)rank * BN;
  const int nk = (P.K + BK - 1) / BK;
  // consumers of CTA 0's multicast release its slots too: 3 arrivals there
  const uint16_t commit_mask = (uint16_t)((1u << rank) | 1u);

  if (threadIdx.x == 0) {
    prefetch_tmap(&P.tmA);
    prefetch_tmap(&P.tmB);
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], rank == 0 ? CL : 1);
    }
    mbar_init(accum, 1);
    fence_mbar_init();
  }
  if (warp == 2) tmem_alloc(tmem_slot, TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();             // peers' barriers exist before any multicast lands
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0 && lane == 0) {
    // hidden rows (CTA 0, which multicasts them) and weight rows are pulled
    // into L2 2*STAGES k-blocks ahead of their load
    auto prefetch = [&](int kb) {
      if (kb < nk) {
        if (rank == 0) tma_prefetch_3d(&P.tmA, kb * BK, m0, 0);
        tma_prefetch_3d(&P.tmB, kb * BK, n0, 0);
      }
    };
    for (int kb = STAGES; kb < 2 * STAGES; ++kb) prefetch(kb);
    bool ok = true;
    for (int kb = 0; kb < nk && ok; ++kb) {
      const int s = kb % STAGES;
      ok = mbar_wait(&empty[s], ((kb / STAGES) & 1) ^ 1, P.status);
      if (!ok) break;
      uint8_t* a = smem + s * STAGE_BYTES;
      mbar_arrive_expect_tx(&full[s], STAGE_BYTES);
      if (rank == 0) tma_load_3d_mc(a, &P.tmA, &full[s], kb * BK, m0, 0, (1u << CL) - 1);
      tma_load_3d(a + A_BYTES, &P.tmB, &full[s], kb * BK, n0, 0);
      prefetch(kb + 2 * STAGES);
    }
    for (int kb = max(0, nk - STAGES); kb < nk; ++kb)
      mbar_wait(&full[kb % STAGES], (kb / STAGES) & 1, P.status);
  } else if (warp == 1 && lane == 0) {
    const uint32_t idesc = idesc_f16(BM, BN, false);
    for (int kb = 0; kb < nk; ++kb) {
      const int s = kb % STAGES;
      if (!mbar_wait(&full[s], (kb / STAGES) & 1, P.status)) break;
      tc_fence_after();
      const uint8_t* a = smem + s * STAGE_BYTES;
      const uint64_t da = smem_desc_sw128(a), db = smem_desc_sw128(a + A_BYTES);
#pragma unroll
      for (int k = 0; k < BK / 16; ++k) mma_f16(tmem, da + 2 * k, db + 2 * k, idesc, (kb | k) != 0);
      mma_commit_mc(&empty[s], commit_mask);
    }
    mma_commit(accum);
  }
  __syncwarp();

  // ---- epilogue: RMSNorm across the cluster, RoPE, scatter to cache slots ----
  const bool have = mbar_wait(accum, 0, P.status);
  tc_fence_after();
  const int r = warp * 32 + lane, m = m0 + r;
  const uint32_t lane_addr = tmem + ((uint32_t)(warp * 32) << 16);
  const int lat_cols = rank < 2 ? BN : 512 - 2 * BN;   // latent columns held here (rest: rope)
  float ss = 0.f;
#pragma unroll 1
  for (int c = 0; c < BN; c += 32) {
    float v[32];
    tmem_ld32(lane_addr + c, v);
    if (c < lat_cols) {
#pragma unroll
      for (int i = 0; i < 32; ++i) ss = fmaf(v[i], v[i], ss);
    }
  }
  red[r] = ss;
  cluster_sync_all();
  float tot = 0.f;
#pragma unroll
  for (int q = 0; q < CL; ++q) tot += ld_cluster_f32(mapa(smem_u32(&red[r]), q));  // same order in all three
  const float rstd = 1.f / sqrtf(tot / 512.f + P.eps);
  const bool row_ok = have && m < P.M;
  long slot = 0;
  int pos = 0;
  if (row_ok) {
    slot = P.slots[m];
    pos = P.positions[m];
  }
  const bool bad_slot = row_ok && (slot < 0 || slot >= P.num_slots);
  const bool bad_pos = row_ok && rank == CL - 1 && (pos < 0 || pos >= P.max_pos);
  if (bad_slot || bad_pos)
    set_status(P.status, (bad_slot ? MLA_DEV_BAD_SLOT : 0) | (bad_pos ? MLA_DEV_BAD_POSITION : 0));
  const bool store = row_ok && !bad_slot && !bad_pos;
  __nv_bfloat16* dst = P.cache + slot * 576 + n0;
#pragma unroll 1
  for (int c = 0; c < lat_cols; c += 32) {
    float v[32];
    tmem_ld32(lane_addr + c, v);
    if (!store) continue;
#pragma unroll
    for (int i = 0; i < 32; i += 8) {
      __nv_bfloat162 h2[4];
#pragma unroll
      for (int u = 0; u < 4; ++u)
        h2[u] = __floats2bfloat162_rn(v[i + 2 * u] * rstd * P.gamma[n0 + c + i + 2 * u],
                                      v[i + 2 * u + 1] * rstd * P.gamma[n0 + c + i + 2 * u + 1]);
      *reinterpret_cast<uint4*>(dst + c + i) = *reinterpret_cast<uint4*>(h2);
    }
  }
  if (rank == CL - 1) {
    // rope columns 512..575 = local 128..191: pair k is (2k, 2k+1) interleaved
    // or (k, k + 32) NeoX, rotated by angle k of the position
    float a[32], b[32];
    tmem_ld32(lane_addr + lat_cols, a);
    tmem_ld32(lane_addr + lat_cols + 32, b);
    if (store) {
      float o[64];
      const float2* cs = P.rope + (long)pos * 32;
#pragma unroll
      for (int k = 0; k < 32; ++k) {
        float x, y;
        if (P.interleaved) {
          x = k < 16 ? a[2 * k] : b[2 * k - 32];
          y = k < 16 ? a[2 * k + 1] : b[2 * k - 31];
        } else {
          x = a[k];
          y = b[k];
        }
        const float2 t = cs[k];
        const float rx = x * t.x - y * t.y, ry = y * t.x + x * t.y;
        if (P.interleaved) { o[2 * k] = rx; o[2 * k + 1] = ry; }
        else { o[k] = rx; o[k + 32] = ry; }
      }
#pragma unroll
      for (int i = 0; i < 64; i += 8) {
        __nv_bfloat162 h2[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) h2[u] = __floats2bfloat162_rn(o[i + 2 * u], o[i + 2 * u + 1]);
        *reinterpret_cast<uint4*>(dst + lat_cols + i) = *reinterpret_cast<uint4*>(h2);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();             // no CTA leaves while a peer may still read its partials
  if (warp == 2) tmem_dealloc(tmem, TMEM_COLS);
}

}  // namespace

mla_status_t kv_append(cudaStream_t st, const mla_handle* h, const __nv_bfloat16* hidden, int M,
                       const int32_t* positions, const int64_t* slots, __nv_bfloat16* cache,
                       long num_slots) {
  const Layout& l = h->lay;
  if (l.rkv != 512 || l.dr != 64)
    return fail(MLA_ERR_UNSUPPORTED, "tcgen05 append: needs kv_lora_rank 512, qk_rope_head_dim 64");
  if (l.D % 8) return fail(MLA_ERR_UNSUPPORTED, "tcgen05 append: hidden_size must be a multiple of 8");
  if (M <= 0) return MLA_OK;
  AppendParams P;
  if (!make_tmap_2d(&P.tmA, false, hidden, M, l.D, l.D, BM) ||
      !make_tmap_2d(&P.tmB, false, h->WA, 576, l.D, l.D, BN))
    return fail(MLA_ERR_CUDA, "tcgen05 append: cuTensorMapEncodeTiled failed");
  P.M = M;
  P.K = l.D;
  P.positions = positions;
  P.slots = slots;
  P.cache = cache;
  P.num_slots = num_slots;
  P.gamma = h->gamma_kv;
  P.rope = h->rope;
  P.max_pos = h->cfg.max_position;
  P.interleaved = h->cfg.rope == MLA_ROPE_INTERLEAVED;
  P.eps = (float)h->cfg.rms_norm_eps;
  P.status = h->status;
  static std::once_flag once;
  std::call_once(once, [] {
    cudaFuncSetAttribute(kv_append_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
  });
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(CL, (M + BM - 1) / BM, 1);
  cfg.blockDim = dim3(THREADS, 1, 1);
  cfg.dynamicSmemBytes = SMEM_BYTES;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CL;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kv_append_tc_kernel, P);
  if (e != cudaSuccess) return cuda_fail(e, "tcgen05 append launch");
  return MLA_OK;
}

}  // namespace tc
}  // namespace mla
