// Latent-cache append on tcgen05 ("MLA (Multi-Head Latent Attention)" blog,
// wrapper forward + do_kv_cache_update / concat_and_cache_mla):
//   kv = hidden @ W_kva^T                     (W_kva: the kv_lora_rank + qk_rope rows)
//   cache[slot] = [RMSNorm(kv[:512]) * gamma | RoPE(kv[512:], position)]   (bf16)
//
// Persistent kernel.  A cluster of 3 CTAs works on 128 token rows at a time
// (a "tile") and loops over tiles: CTA c computes output columns
// [192c, 192c + 192) of the tile's rows.  Every CTA streams its own operands
// with TMA: the tile's hidden-state rows (the three CTAs of a cluster read the
// same rows, so two of the three reads hit L2) and its 192 weight rows (read
// by every cluster, L2-resident).  One ring stage holds KBS consecutive
// 64-wide k-blocks of both operands, each brought by a single chunked copy.
//
// Warps 0 and 6 stream the ring (hidden states and weights: a TMA copy keeps
// its issuing thread for about 550 cycles whatever its size, while copies of
// different warps proceed side by side), warp 1 issues the MMAs into one of
// two tensor-memory accumulators (192 columns each), warps 2-5 run the epilogue of the
// previous tile meanwhile: per row the sum of squares of its latent columns,
// exchanged with the two other CTAs of the cluster through asynchronous
// distributed-shared-memory stores (counted on an mbarrier) and added in the
// same order everywhere; then normalisation, RoPE (CTA 2 holds the 64 rope
// columns); each epilogue warp stages its own 32 rows 64 columns at a time in
// shared memory and writes them to the rows' cache slots as whole 128-byte
// pieces.
#include "append_tc.cuh"

#include <mutex>

#include "gemm_tc.cuh"
#include "tc_ptx.cuh"

namespace mla {
namespace tc {
namespace {

#ifndef MLA_APPEND_KBS
#define MLA_APPEND_KBS 1
#endif
constexpr int BM = 128, BN = 192, BK = 64;
constexpr int KBS = MLA_APPEND_KBS;               // k-blocks per ring stage (one copy per operand)
constexpr int STAGES = KBS == 1 ? 5 : KBS == 2 ? 2 : 1;
constexpr int CL = 3;                             // cluster: the 3 column CTAs of a row tile
constexpr int THREADS = 224;                      // TMA (A), MMA, 4 epilogue warps, TMA (B)
constexpr int EPI = 128;                          // epilogue threads
constexpr int A_BYTES = KBS * BM * BK * 2, B_BYTES = KBS * BN * BK * 2;
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int GC = 64;                            // columns staged at a time
constexpr int OUT_PITCH = GC * 2 + 16;            // staged output row (bytes), bank-conflict free
constexpr int OFF_OUT = STAGES * STAGE_BYTES;     // per epilogue warp: 32 staged rows [32][OUT_PITCH]
constexpr int OFF_RED = OFF_OUT + BM * OUT_PITCH; // partial sums of squares [2][CL][BM]
constexpr int OFF_GAM = OFF_RED + 2 * CL * BM * 4;  // this CTA's kv_a_layernorm gains [BN]
constexpr int OFF_BAR = OFF_GAM + BN * 4;
constexpr int SMEM_BYTES = 1024 + OFF_BAR + 256;
constexpr uint32_t TMEM_COLS = 512, ACC_STRIDE = 256;   // two accumulators of BN columns
static_assert(SMEM_BYTES <= 232448, "shared memory");

struct AppendParams {
  CUtensorMap tmA;            // hidden [M, D], chunked view, box 128 rows x KBS k-blocks
  CUtensorMap tmB;            // W_kva [576, D], chunked view, box 192 rows x KBS k-blocks
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

struct Bars {
  uint64_t full[STAGES], empty[STAGES];   // ring: both copies landed / this CTA's MMAs done with the slot
  uint64_t acc_full[2], acc_empty[2];     // accumulator b written (MMA) / read (epilogue)
  uint64_t red_full[2];                   // the two peers' partial sums of tile parity b landed
  uint64_t red_free[2];                   // the two peers have read what this CTA sent them
  uint64_t drain;                         // every MMA of the CTA complete
  uint32_t tmem_slot;
  int abort;
};
static_assert(sizeof(Bars) <= 256, "barrier block");

// Bounded waits that give up at once after any earlier timeout of this CTA.
__device__ __forceinline__ bool wait_bar(Bars* B, uint64_t* bar, uint32_t parity, uint32_t* st) {
  if (*(volatile int*)&B->abort) return false;
  if (mbar_wait_cluster(bar, parity, st)) return true;
  B->abort = 1;
  return false;
}

__device__ __forceinline__ void st_async_b32(uint32_t remote_addr, float v, uint32_t remote_bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];"
               ::"r"(remote_addr), "r"(__float_as_uint(v)), "r"(remote_bar) : "memory");
}

__global__ void __launch_bounds__(THREADS, 1) kv_append_tc_kernel(const __grid_constant__ AppendParams P) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  Bars* B = (Bars*)(smem + OFF_BAR);
  float* red = (float*)(smem + OFF_RED);
  float* gam = (float*)(smem + OFF_GAM);

  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  const int c = (int)cluster_ctarank();              // column group (== blockIdx.x)
  const int n0 = c * BN;
  const int nk = (P.K + BK - 1) / BK;
  const int ns = (nk + KBS - 1) / KBS;               // ring stages per tile
  const int n_ct = (P.M + BM - 1) / BM;              // row tiles of 128
  const int cid = blockIdx.y, ncl = gridDim.y;

  if (tid == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&B->full[s], 2);          // one arrival per producer warp
      mbar_init(&B->empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&B->acc_full[b], 1);
      mbar_init(&B->acc_empty[b], EPI);
      mbar_init(&B->red_full[b], 1);
      mbar_init(&B->red_free[b], 2 * (EPI / 32));   // 4 warps of each of the two peers
    }
    mbar_init(&B->drain, 1);
    B->abort = 0;
    fence_mbar_init();
    // the first use of each partial-sum buffer expects both peers' rows
    for (int b = 0; b < 2; ++b) mbar_arrive_expect_tx(&B->red_full[b], 2 * BM * 4);
  }
  for (int i = tid; i < BN; i += THREADS) gam[i] = n0 + i < 512 ? P.gamma[n0 + i] : 0.f;
  if (warp == 1) tmem_alloc(&B->tmem_slot, TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();             // peers' barriers exist before any remote store
  tc_fence_after();
  const uint32_t tmem = B->tmem_slot;
  if (tid == 0) pdl_trigger();
  pdl_wait();

  if (warp == 0 || warp == 6) {
    if (lane == 0) {
      // ---- TMA producers: warp 0 the hidden-state rows, warp 6 the weights ----
      const bool is_a = warp == 0;
      const CUtensorMap* map = is_a ? &P.tmA : &P.tmB;
      prefetch_tmap(map);
      int g = 0;
      bool ok = true;
      for (int ct = cid; ct < n_ct && ok; ct += ncl) {
        const int row = is_a ? ct * BM : n0;
        for (int ks = 0; ks < ns; ++ks, ++g) {
          const int s = g % STAGES;
          if (!wait_bar(B, &B->empty[s], ((g / STAGES) & 1) ^ 1, P.status)) { ok = false; break; }
          uint8_t* a = smem + s * STAGE_BYTES;
          mbar_arrive_expect_tx(&B->full[s], is_a ? A_BYTES : B_BYTES);
          tma_load_3d(is_a ? a : a + A_BYTES, map, &B->full[s], 0, row, ks * KBS);
        }
      }
      // every copy into this CTA has landed before it may exit
      for (int i = max(0, g - STAGES); i < g; ++i) mbar_wait(&B->full[i % STAGES], (i / STAGES) & 1, P.status);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---- MMA issuer ----
      const uint32_t idesc = idesc_f16(BM, BN, false);
      int g = 0, i = 0;
      bool ok = true;
      for (int ct = cid; ct < n_ct && ok; ct += ncl, ++i) {
        const int b = i & 1;
        if (!wait_bar(B, &B->acc_empty[b], ((i >> 1) & 1) ^ 1, P.status)) break;   // epilogue done with it
        tc_fence_after();
        const uint32_t d = tmem + b * ACC_STRIDE;
        for (int ks = 0; ks < ns; ++ks, ++g) {
          const int s = g % STAGES;
          if (!wait_bar(B, &B->full[s], (g / STAGES) & 1, P.status)) { ok = false; break; }
          tc_fence_after();
          const uint8_t* a = smem + s * STAGE_BYTES;
#pragma unroll
          for (int i = 0; i < KBS; ++i) {
            if (ks * KBS + i >= nk) break;      // k-blocks past K were zero-filled by TMA
            const uint64_t da = smem_desc_sw128(a + i * BM * BK * 2);
            const uint64_t db = smem_desc_sw128(a + A_BYTES + i * BN * BK * 2);
#pragma unroll
            for (int k = 0; k < BK / 16; ++k) mma_f16(d, da + 2 * k, db + 2 * k, idesc, (ks | i | k) != 0);
          }
          mma_commit(&B->empty[s]);
        }
        if (ok) mma_commit(&B->acc_full[b]);
      }
      // no MMA of this CTA may still run when its tensor memory is freed
      mma_commit(&B->drain);
      mbar_wait(&B->drain, 0, P.status);
    }
  } else {
    // ---- epilogue (warps 2-5): thread = accumulator row = TMEM lane ----
    const int q = warp % 4, r = q * 32 + lane;
    const uint32_t lane_off = (uint32_t)(q * 32) << 16;
    const int lat_cols = c < 2 ? BN : 512 - 2 * BN;    // latent columns held here (rest: rope)
    uint8_t* wst = smem + OFF_OUT + q * 32 * OUT_PITCH;   // this warp's staged rows
    uint4* orow = reinterpret_cast<uint4*>(wst + lane * OUT_PITCH);
    int i = 0;
    for (int ct = cid; ct < n_ct; ct += ncl, ++i) {
      const int b = i & 1;
      const uint32_t ph = (i >> 1) & 1;
      const int m = ct * BM + r;
      // waits that give up leave garbage, but every thread still runs the
      // same sequence of epilogue barriers
      const bool have = wait_bar(B, &B->acc_full[b], ph, P.status);
      tc_fence_after();
      const uint32_t lane_addr = tmem + b * ACC_STRIDE + lane_off;
      float ss = 0.f;
#pragma unroll 1
      for (int col = 0; col < lat_cols; col += 32) {
        float v[32];
        tmem_ld32(lane_addr + col, v);
#pragma unroll
        for (int k = 0; k < 32; ++k) ss = fmaf(v[k], v[k], ss);
      }
      // partial sum of squares: own slot locally, the two peers' by async stores
      wait_bar(B, &B->red_free[b], ph ^ 1, P.status);
      float* rb = red + b * CL * BM;
      rb[c * BM + r] = ss;
#pragma unroll
      for (int k = 1; k < CL; ++k) {
        const uint32_t peer = (uint32_t)((c + k) % CL);
        st_async_b32(mapa(smem_u32(&rb[c * BM + r]), peer), ss, mapa(smem_u32(&B->red_full[b]), peer));
      }
      wait_bar(B, &B->red_full[b], ph, P.status);
      const float tot = (rb[r] + rb[BM + r]) + rb[2 * BM + r];     // same order in all three
      // this warp is done reading the peers' partials of parity b
      __syncwarp();
      if (lane == 0) {
#pragma unroll
        for (int k = 1; k < CL; ++k) mbar_arrive_remote(mapa(smem_u32(&B->red_free[b]), (uint32_t)((c + k) % CL)));
      }
      if (r == 0) mbar_arrive_expect_tx(&B->red_full[b], 2 * BM * 4);   // armed for tile i + 2
      const float rstd = 1.f / sqrtf(tot / 512.f + P.eps);
      const bool row_ok = have && m < P.M;
      long slot = 0;
      int pos = 0;
      if (row_ok) {
        slot = P.slots[m];
        pos = P.positions[m];
      }
      const bool bad_slot = row_ok && (slot < 0 || slot >= P.num_slots);
      const bool bad_pos = row_ok && c == CL - 1 && (pos < 0 || pos >= P.max_pos);
      if (bad_slot || bad_pos)
        set_status(P.status, (bad_slot ? MLA_DEV_BAD_SLOT : 0) | (bad_pos ? MLA_DEV_BAD_POSITION : 0));
      const bool store = row_ok && !bad_slot && !bad_pos;
      const long my_slot = store ? slot : -1;
      // 64 columns at a time: the rows' bf16 values -> this warp's staging
      // rows -> global, lanes 8k .. 8k+7 writing one 128-byte row piece
#pragma unroll 1
      for (int col = 0; col < BN; col += GC) {
        float v[GC];
        tmem_ld32(lane_addr + col, v);
        tmem_ld32(lane_addr + col + 32, v + 32);
        if (col < lat_cols) {
#pragma unroll
          for (int k = 0; k < GC; ++k) v[k] *= rstd * gam[col + k];
        } else {
          // rope columns 512..575 (local 128..191 of column CTA 2): pair k is
          // (2k, 2k+1) interleaved or (k, k + 32) NeoX, rotated by angle k
          const float2* cs = P.rope + (long)(store ? pos : 0) * 32;
          float o[GC];
#pragma unroll
          for (int k = 0; k < 32; ++k) {
            const float x = P.interleaved ? v[2 * k] : v[k];
            const float y = P.interleaved ? v[2 * k + 1] : v[k + 32];
            const float2 t = cs[k];
            const float rx = x * t.x - y * t.y, ry = y * t.x + x * t.y;
            if (P.interleaved) { o[2 * k] = rx; o[2 * k + 1] = ry; }
            else { o[k] = rx; o[k + 32] = ry; }
          }
#pragma unroll
          for (int k = 0; k < GC; ++k) v[k] = o[k];
        }
#pragma unroll
        for (int k = 0; k < GC; k += 8) {
          __nv_bfloat162 h2[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) h2[u] = __floats2bfloat162_rn(v[k + 2 * u], v[k + 2 * u + 1]);
          orow[k / 8] = *reinterpret_cast<uint4*>(h2);
        }
        __syncwarp();
#pragma unroll
        for (int it = 0; it < 8; ++it) {
          const int row = 4 * it + lane / 8, piece = lane % 8;
          const long sl = __shfl_sync(0xffffffffu, my_slot, row);
          if (sl >= 0)
            reinterpret_cast<uint4*>(P.cache + sl * 576 + n0 + col)[piece] =
                reinterpret_cast<const uint4*>(wst + row * OUT_PITCH)[piece];
        }
        __syncwarp();                 // the staging rows are rewritten by the next group
      }
      // accumulator b may be overwritten by tile i + 2
      tc_fence_before();
      mbar_arrive(&B->acc_empty[b]);
    }
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();             // no CTA leaves while a peer may still store to it or arrive on its barriers
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, TMEM_COLS);
}

}  // namespace

mla_status_t kv_append(cudaStream_t st, const mla_handle* h, const __nv_bfloat16* hidden, int M,
                       const int32_t* positions, const int64_t* slots, __nv_bfloat16* cache,
                       long num_slots, bool pdl) {
  const Layout& l = h->lay;
  if (l.rkv != 512 || l.dr != 64)
    return fail(MLA_ERR_UNSUPPORTED, "tcgen05 append: needs kv_lora_rank 512, qk_rope_head_dim 64");
  if (l.D % 8) return fail(MLA_ERR_UNSUPPORTED, "tcgen05 append: hidden_size must be a multiple of 8");
  if (M <= 0) return MLA_OK;
  AppendParams P;
  if (!make_tmap_chunked(&P.tmA, false, hidden, M, l.D, l.D, BM, KBS) ||
      !make_tmap_chunked(&P.tmB, false, h->WA, 576, l.D, l.D, BN, KBS))
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
  // persistent: as many clusters as fit on the GPU at once, at most one per cluster tile
  static std::once_flag once_occ;
  static int max_clusters = 0;
  std::call_once(once_occ, [] {
    cudaLaunchConfig_t c = {};
    c.gridDim = dim3(CL, 1, 1);
    c.blockDim = dim3(THREADS, 1, 1);
    c.dynamicSmemBytes = SMEM_BYTES;
    cudaLaunchAttribute a[1];
    a[0].id = cudaLaunchAttributeClusterDimension;
    a[0].val.clusterDim.x = CL;
    a[0].val.clusterDim.y = 1;
    a[0].val.clusterDim.z = 1;
    c.attrs = a;
    c.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kv_append_tc_kernel, &c) != cudaSuccess || n <= 0) {
      (void)cudaGetLastError();
      n = 16;
    }
    max_clusters = n;
  });
  const int n_ct = (M + BM - 1) / BM;
  const int ncl = n_ct < max_clusters ? n_ct : max_clusters;
  Launch L(dim3(CL, ncl, 1), dim3(THREADS), SMEM_BYTES, st, pdl, dim3(CL, 1, 1));
  const cudaError_t e = cudaLaunchKernelEx(&L.cfg, kv_append_tc_kernel, P);
  if (e != cudaSuccess) return cuda_fail(e, "tcgen05 append launch");
  return MLA_OK;
}

}  // namespace tc
}  // namespace mla
