// Latent-cache append on tcgen05 ("MLA (Multi-Head Latent Attention)" blog,
// wrapper forward + do_kv_cache_update / concat_and_cache_mla):
//   kv = hidden @ W_kva^T                     (W_kva: the kv_lora_rank + qk_rope rows)
//   cache[slot] = [RMSNorm(kv[:512]) * gamma | RoPE(kv[512:], position)]   (bf16)
//
// A cluster of 3 x 2 CTAs owns 256 token rows: CTA (c, r) computes output
// columns [192c, 192c + 192) of rows [128r, 128r + 128) in tensor memory.
// Every 128 x 64 slice of hidden states is multicast to the three CTAs of its
// row group and every 192 x 64 slice of weights to the two CTAs of its column
// group, so each cluster reads its hidden rows and each weight slice once.  A
// TMA copy costs about the same SM time whatever its size, so the copies of a
// k-block are issued by different CTAs in turn (hidden: CTA c = kb mod 3 of
// the row group, weights: CTA r = kb mod 2 of the column group), each SM
// issuing less than one copy per k-block.  In the epilogue every CTA adds the
// squares of its latent columns per row, the three partial sums of a row
// group are exchanged through distributed shared memory and added in the same
// order everywhere, and each CTA normalises, rotates (column CTA 2 holds the
// 64 rope columns) and stores its part of every row straight to the row's
// cache slot.
#include "append_tc.cuh"

#include <mutex>

#include "gemm_tc.cuh"
#include "tc_ptx.cuh"

namespace mla {
namespace tc {
namespace {

constexpr int BM = 128, BN = 192, BK = 64, THREADS = 128, STAGES = 5;
constexpr int CL = 3, CR = 2, NCTA = CL * CR;     // cluster: 3 column CTAs x 2 row groups
constexpr int A_BYTES = BM * BK * 2, B_BYTES = BN * BK * 2, STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int OFF_BAR = STAGES * STAGE_BYTES;
constexpr int SMEM_BYTES = 1024 + OFF_BAR + 2048;
constexpr uint32_t TMEM_COLS = 256;
constexpr int OUT_PITCH = BN * 2 + 16;            // staged output row (bytes), bank-conflict free
static_assert(BM * OUT_PITCH + BM * 8 <= OFF_BAR, "output staging fits in the pipeline stages");

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
  float* gam = red + BM;                           // this CTA's kv_a_layernorm gains [BN]

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const uint32_t rank = cluster_ctarank();         // c + 3 r
  const int c = (int)rank % CL, rg = (int)rank / CL; // column group (== blockIdx.x), row group
  const int m0 = blockIdx.y * BM, n0 = c * BN;
  const int nk = (P.K + BK - 1) / BK;
  // a slot is refilled once all six CTAs are done with it
  const uint16_t all_mask = (uint16_t)((1u << NCTA) - 1);
  const uint16_t row_mask = (uint16_t)(0x7u << (CL * rg));            // CTAs of this row group
  const uint16_t col_mask = (uint16_t)((1u << c) | (1u << (c + CL)));  // CTAs of this column group

  if (threadIdx.x == 0) {
    prefetch_tmap(&P.tmA);
    prefetch_tmap(&P.tmB);
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], NCTA);
    }
    mbar_init(accum, 1);
    fence_mbar_init();
  }
  if (warp == 2) tmem_alloc(tmem_slot, TMEM_COLS);
  for (int i = threadIdx.x; i < BN; i += THREADS) gam[i] = n0 + i < 512 ? P.gamma[n0 + i] : 0.f;
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();             // peers' barriers exist before any multicast lands
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  if (threadIdx.x == 0) pdl_trigger();
  pdl_wait();

  if (warp == 0 && lane == 0) {
    // the hidden rows of a k-block are pulled into L2 2*STAGES k-blocks ahead
    // of their load, by the CTA that will load them
    auto prefetch = [&](int kb) {
      if (kb < nk && kb % CL == c) tma_prefetch_3d(&P.tmA, kb * BK, m0, 0);
    };
    for (int kb = STAGES; kb < 2 * STAGES; ++kb) prefetch(kb);
    bool ok = true;
    for (int kb = 0; kb < nk && ok; ++kb) {
      const int s = kb % STAGES;
      ok = mbar_wait_cluster(&empty[s], ((kb / STAGES) & 1) ^ 1, P.status);
      if (!ok) break;
      uint8_t* a = smem + s * STAGE_BYTES;
      mbar_arrive_expect_tx(&full[s], STAGE_BYTES);
      if (kb % CL == c) tma_load_3d_mc(a, &P.tmA, &full[s], kb * BK, m0, 0, row_mask);
      if (kb % CR == rg) tma_load_3d_mc(a + A_BYTES, &P.tmB, &full[s], kb * BK, n0, 0, col_mask);
      prefetch(kb + 2 * STAGES);
    }
    for (int kb = max(0, nk - STAGES); kb < nk; ++kb)
      mbar_wait_cluster(&full[kb % STAGES], (kb / STAGES) & 1, P.status);
  } else if (warp == 1 && lane == 0) {
    const uint32_t idesc = idesc_f16(BM, BN, false);
    for (int kb = 0; kb < nk; ++kb) {
      const int s = kb % STAGES;
      if (!mbar_wait_cluster(&full[s], (kb / STAGES) & 1, P.status)) break;
      tc_fence_after();
      const uint8_t* a = smem + s * STAGE_BYTES;
      const uint64_t da = smem_desc_sw128(a), db = smem_desc_sw128(a + A_BYTES);
#pragma unroll
      for (int k = 0; k < BK / 16; ++k) mma_f16(tmem, da + 2 * k, db + 2 * k, idesc, (kb | k) != 0);
      mma_commit_mc(&empty[s], all_mask);
    }
    mma_commit(accum);
  }
  __syncwarp();

  // ---- epilogue: RMSNorm across the cluster, RoPE, rows to cache slots ----
  const bool have = mbar_wait(accum, 0, P.status);
  tc_fence_after();
  const int r = warp * 32 + lane, m = m0 + r;
  const uint32_t lane_addr = tmem + ((uint32_t)(warp * 32) << 16);
  const int lat_cols = c < 2 ? BN : 512 - 2 * BN;      // latent columns held here (rest: rope)
  float ss = 0.f;
#pragma unroll 1
  for (int col = 0; col < BN; col += 32) {
    float v[32];
    tmem_ld32(lane_addr + col, v);
    if (col < lat_cols) {
#pragma unroll
      for (int i = 0; i < 32; ++i) ss = fmaf(v[i], v[i], ss);
    }
  }
  red[r] = ss;
  cluster_sync_all();
  float tot = 0.f;
#pragma unroll
  for (int q = 0; q < CL; ++q) tot += ld_cluster_f32(mapa(smem_u32(&red[r]), CL * rg + q));  // same order in all three
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
  // the row's 192 bf16 outputs go to shared memory first (the pipeline stages
  // are free once the accumulator is complete); rows then leave as whole
  // 384-byte segments written by a warp together
  uint8_t* out_tile = smem;                                  // [BM][OUT_PITCH]
  long* out_slot = (long*)(smem + BM * OUT_PITCH);           // [BM], -1 = not stored
  uint4* orow = reinterpret_cast<uint4*>(out_tile + r * OUT_PITCH);
#pragma unroll 1
  for (int col = 0; col < lat_cols; col += 32) {
    float v[32];
    tmem_ld32(lane_addr + col, v);
#pragma unroll
    for (int i = 0; i < 32; i += 8) {
      __nv_bfloat162 h2[4];
#pragma unroll
      for (int u = 0; u < 4; ++u)
        h2[u] = __floats2bfloat162_rn(v[i + 2 * u] * rstd * gam[col + i + 2 * u],
                                      v[i + 2 * u + 1] * rstd * gam[col + i + 2 * u + 1]);
      orow[(col + i) / 8] = *reinterpret_cast<uint4*>(h2);
    }
  }
  if (c == CL - 1) {
    // rope columns 512..575 = local 128..191: pair k is (2k, 2k+1) interleaved
    // or (k, k + 32) NeoX, rotated by angle k of the position
    float a[32], b[32];
    tmem_ld32(lane_addr + lat_cols, a);
    tmem_ld32(lane_addr + lat_cols + 32, b);
    float o[64];
    const float2* cs = P.rope + (long)(store ? pos : 0) * 32;
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
      orow[(lat_cols + i) / 8] = *reinterpret_cast<uint4*>(h2);
    }
  }
  out_slot[r] = store ? slot : -1;
  __syncthreads();
  // warp w writes rows 32w .. 32w+31, lanes 0..23 one 16-byte piece each
#pragma unroll 1
  for (int i = 0; i < 32; ++i) {
    const int row = warp * 32 + i;
    const long sl = out_slot[row];
    if (sl >= 0 && lane < BN * 2 / 16)
      reinterpret_cast<uint4*>(P.cache + sl * 576 + n0)[lane] =
          reinterpret_cast<const uint4*>(out_tile + row * OUT_PITCH)[lane];
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();             // no CTA leaves while a peer may still read its partials
  if (warp == 2) tmem_dealloc(tmem, TMEM_COLS);
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
  Launch L(dim3(CL, CR * ((M + CR * BM - 1) / (CR * BM)), 1), dim3(THREADS), SMEM_BYTES, st, pdl,
           dim3(CL, CR, 1));
  const cudaError_t e = cudaLaunchKernelEx(&L.cfg, kv_append_tc_kernel, P);
  if (e != cudaSuccess) return cuda_fail(e, "tcgen05 append launch");
  return MLA_OK;
}

}  // namespace tc
}  // namespace mla
