// tcgen05 latent attention of the MLA draft layer ("MLA (Multi-Head Latent
// Attention)" blog, forward_mqa / decode_attention_fwd: one shared 576-wide
// latent KV head; queries absorbed into the latent space; output in the
// 512-wide latent value space).
//
// Work unit: one query block and 128 consecutive rows of Q_abs (rows are
// (token, head) pairs, token-major), handled by a cluster of two CTAs.  The
// 128 x 512 fp32 output accumulator does not fit one SM's tensor memory next
// to a score tile, so CTA r keeps value columns [256r, 256r+256) in TMEM
// (256 columns) plus a 128 x 64 score tile (64 columns).  The score reduction
// over the 576 latent dims is split between the pair: CTA 0 owns dims
// 0..255 and the rope dims 512..575, CTA 1 owns dims 256..511, which are also
// exactly the value dims each needs, so every cache byte is loaded once per
// pair.  Per 64-key tile:
//   MMA warp : S_r = Q_r K_r^T over its own dims (tcgen05, TMEM)
//   softmax  : read S_r, send it to the peer through DSMEM, add the peer's
//              partial (same order in both CTAs, so both see identical
//              scores), mask by logical position, online softmax in fp32
//              (exp2 domain, rescale of the TMEM accumulator only when the
//              running max grows by more than 2^8), write P (bf16) to smem
//   MMA warp : O_r += P V_r (V read MN-major straight from the staged tile)
// Warps 0-3 (thread = accumulator row / TMEM lane) run the softmax and the
// epilogue, warp 4 streams Q and KV tiles with TMA, warp 5 issues MMAs.
#include "attn_tc.cuh"

#include <mutex>

#include "tc_ptx.cuh"

namespace mla {
namespace tc {
namespace {

constexpr int QROWS = 128, KT = 64, DCH = 64;    // query rows, keys per tile, dims per chunk
constexpr int THREADS = 192;
constexpr int MAX_CH = 5;                         // dim chunks held by CTA 0 (4 latent + rope)
constexpr int Q_CH_BYTES = QROWS * DCH * 2;       // 16 KiB
constexpr int KV_CH_BYTES = KT * DCH * 2;         // 8 KiB
constexpr int KV_STAGE_BYTES = MAX_CH * KV_CH_BYTES;
constexpr int OFF_Q = 0;
constexpr int OFF_KV = OFF_Q + MAX_CH * Q_CH_BYTES;
constexpr int OFF_P = OFF_KV + 2 * KV_STAGE_BYTES;
constexpr int OFF_X = OFF_P + QROWS * KT * 2;
constexpr int OFF_BAR = OFF_X + QROWS * KT * 4;
constexpr int SMEM_BYTES = 1024 + OFF_BAR + 256;
constexpr uint32_t TMEM_COLS = 512, TM_O = 0, TM_S = 256;   // S double-buffered: 256, 320
constexpr float RESCALE_LOG2 = 8.f;               // lazy rescale threshold (factor 256)

struct Bars {
  uint64_t q_full, kv_full[2], kv_empty[2], s_full[2], s_free[2], p_full, o_done, x_full, x_empty;
  uint32_t tmem_slot;
  int abort;
};

__device__ __forceinline__ int dim_chunk(int rank, int i) {
  return rank == 0 ? (i < 4 ? i : 8) : 4 + i;    // global 64-dim chunk of local chunk i
}

}  // namespace
}  // namespace tc
}  // namespace mla

namespace mla {
namespace tc {
namespace {

// Bounded waits that give up at once after any earlier timeout of this CTA.
__device__ __forceinline__ bool wait_local(Bars* B, uint64_t* bar, uint32_t parity, uint32_t* st) {
  if (*(volatile int*)&B->abort) return false;
  if (mbar_wait(bar, parity, st)) return true;
  B->abort = 1;
  return false;
}
__device__ __forceinline__ bool wait_peer(Bars* B, uint64_t* bar, uint32_t parity, uint32_t* st) {
  if (*(volatile int*)&B->abort) return false;
  if (mbar_wait_cluster(bar, parity, st)) return true;
  B->abort = 1;
  return false;
}

// 2^x by the hardware approximation (relative error ~2^-22, far below the
// bf16 rounding P gets); 2^-inf = 0.
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Named barrier of the 128 softmax threads (barrier 0 is __syncthreads).
__device__ __forceinline__ void softmax_bar_sync() {
  asm volatile("bar.sync 1, 128;" ::: "memory");
}

// Warps 0-3: thread r owns accumulator row r (TMEM lane r) of the tile.
__device__ __forceinline__ void softmax_and_store(const AttnParams& P, Bars* B, uint8_t* smem,
                                                  uint32_t tmem, uint32_t rank, uint32_t peer,
                                                  int b, int qt, long row0, int kvl, int W,
                                                  int j_lo, int nt) {
  const int r = threadIdx.x;
  const uint32_t lane_base = (uint32_t)((r / 32) * 32) << 16;
  const int row_in_block = qt * QROWS + r;
  const int tok = row_in_block / P.H, head = row_in_block % P.H;
  const long m = (long)b * P.T + tok;
  const int p = P.positions[m];
  const bool qv = P.q_visible ? P.q_visible[m] != 0 : true;
  // the keys this query sees form one interval [vlo, vhi): j < kv_len and, for
  // a sliding window, p - j < W; a fully masked query sees none
  const int vlo = W > 0 ? max(0, p - W + 1) : 0;
  const int vhi = qv ? kvl : 0;
  float* xrow = (float*)(smem + OFF_X) + r * KT;
  const uint32_t peer_xrow = mapa(smem_u32(xrow), peer);
  const uint32_t peer_xfull = mapa(smem_u32(&B->x_full), peer);
  const uint32_t peer_xempty = mapa(smem_u32(&B->x_empty), peer);
  uint8_t* prow = smem + OFF_P + r * 128;
  float mrun = -INFINITY, lsum = 0.f;
  int cnt = 0, first = -1, last = -1;
  for (int t = 0; t < nt; ++t) {
    const int j0 = j_lo + t * KT;
    float s[KT];
    const uint32_t sbuf = tmem + TM_S + 64 * (t & 1) + lane_base;
    wait_local(B, &B->s_full[t & 1], (t >> 1) & 1, P.status);
    tc_fence_after();
    // exchange the partial scores with the peer CTA (its buffer is free once
    // it has read the previous tile)
    tmem_ld32(sbuf, s);
    wait_local(B, &B->x_empty, (t & 1) ^ 1, P.status);
#pragma unroll
    for (int i = 0; i < 32; i += 4) st_cluster_v4(peer_xrow + 4 * i, s[i], s[i + 1], s[i + 2], s[i + 3]);
    tmem_ld32(sbuf + 32, s + 32);
    tc_fence_before();
    mbar_arrive(&B->s_free[t & 1]);
#pragma unroll
    for (int i = 32; i < KT; i += 4) st_cluster_v4(peer_xrow + 4 * i, s[i], s[i + 1], s[i + 2], s[i + 3]);
    // all 128 rows stored, then one cluster-scope release carries them to the peer
    softmax_bar_sync();
    if (r == 0) mbar_arrive_remote(peer_xfull);
    wait_peer(B, &B->x_full, t & 1, P.status);
#pragma unroll
    for (int i = 0; i < KT; i += 4) {
      const float4 x = *reinterpret_cast<const float4*>(xrow + i);
      const float xs[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
      for (int u = 0; u < 4; ++u) s[i + u] = rank == 0 ? s[i + u] + xs[u] : xs[u] + s[i + u];
    }
    softmax_bar_sync();
    if (r == 0) mbar_arrive_remote(peer_xempty);   // every row read: the peer may write again
    // mask by logical position, scale into the exp2 domain
    const int lo = max(vlo - j0, 0), hi = min(vhi - j0, KT);   // visible columns [lo, hi)
    if (hi > lo) {
      cnt += hi - lo;
      if (first < 0) first = j0 + lo;
      last = j0 + hi - 1;
    }
    float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
    for (int i = 0; i < KT; ++i) {
      s[i] = (i >= lo && i < hi) ? s[i] * P.scale_log2 : -INFINITY;
      mx4[i & 3] = fmaxf(mx4[i & 3], s[i]);
    }
    const float tmax = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3]));
    const bool grow = tmax > mrun + RESCALE_LOG2;
    const float m_new = grow ? tmax : mrun;
    const float mref = m_new == -INFINITY ? 0.f : m_new;      // all masked so far: P = 0
    float ps4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int i = 0; i < KT; ++i) {
      s[i] = fast_exp2(s[i] - mref);
      ps4[i & 3] += s[i];
    }
    const float psum = (ps4[0] + ps4[1]) + (ps4[2] + ps4[3]);
    // the previous P.V has finished: P may be overwritten and O rescaled
    if (t > 0) wait_local(B, &B->o_done, (t - 1) & 1, P.status);
    tc_fence_after();
    const float alpha = (grow && mrun != -INFINITY) ? exp2f(mrun - m_new) : 1.f;
    if (t > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll 1
      for (int c = 0; c < 256; c += 32) {
        float o[32];
        tmem_ld32(tmem + TM_O + lane_base + c, o);
#pragma unroll
        for (int i = 0; i < 32; ++i) o[i] *= alpha;
        tmem_st32(tmem + TM_O + lane_base + c, o);
      }
    }
    lsum = lsum * alpha + psum;
    mrun = m_new;
    // value rows of keys past kv_len may hold anything: zero them (last tile)
    if (j0 + KT > kvl) {
      uint8_t* stage = smem + OFF_KV + (t & 1) * KV_STAGE_BYTES;
      const int z0 = max(0, kvl - j0), pieces = (KT - z0) * 4 * 8;
      for (int idx = r; idx < pieces; idx += QROWS) {
        const int key = z0 + idx / 32, ch = (idx % 32) / 8, q = idx % 8;
        *reinterpret_cast<uint4*>(stage + ch * KV_CH_BYTES + key * 128 + q * 16) = make_uint4(0, 0, 0, 0);
      }
    }
    // P row in bf16, 128-byte-swizzled K-major layout (16-byte chunk q of row r at q ^ (r % 8))
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      __nv_bfloat162 h2[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) h2[u] = __floats2bfloat162_rn(s[8 * q + 2 * u], s[8 * q + 2 * u + 1]);
      *reinterpret_cast<uint4*>(prow + ((q ^ (r & 7)) * 16)) = *reinterpret_cast<uint4*>(h2);
    }
    fence_proxy_async_smem();
    tc_fence_before();
    mbar_arrive(&B->p_full);
  }
  // epilogue: O_r / l -> fp16 latent output columns [256 rank, 256 rank + 256)
  if (nt > 0) wait_local(B, &B->o_done, (nt - 1) & 1, P.status);
  tc_fence_after();
  const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
  const bool any = nt > 0 && lsum > 0.f;
  if (P.splits == 1) {
    __half* dst = P.o_lat + (row0 + r) * 512 + rank * 256;
#pragma unroll 1
    for (int c = 0; c < 256; c += 32) {
      float o[32];
      if (nt > 0) tmem_ld32(tmem + TM_O + lane_base + c, o);
#pragma unroll
      for (int i = 0; i < 32; i += 8) {
        __half2 h2[4];
#pragma unroll
        for (int u = 0; u < 4; ++u)
          h2[u] = any ? __floats2half2_rn(o[i + 2 * u] * inv, o[i + 2 * u + 1] * inv)
                      : __floats2half2_rn(0.f, 0.f);
        *reinterpret_cast<uint4*>(dst + c + i) = *reinterpret_cast<uint4*>(h2);
      }
    }
  } else {
    // normalised partial output and its log2-sum-exp, merged by merge_splits()
    const long prow = (long)blockIdx.y * P.rows + row0 + r;
    float* dst = P.o_part + prow * 512 + rank * 256;
#pragma unroll 1
    for (int c = 0; c < 256; c += 32) {
      float o[32];
      if (nt > 0) tmem_ld32(tmem + TM_O + lane_base + c, o);
#pragma unroll
      for (int i = 0; i < 32; i += 4)
        *reinterpret_cast<float4*>(dst + c + i) =
            any ? make_float4(o[i] * inv, o[i + 1] * inv, o[i + 2] * inv, o[i + 3] * inv)
                : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    if (rank == 0) P.lse_part[prow] = any ? mrun + log2f(lsum) : -INFINITY;
  }
  if (P.vis_stats && rank == 0 && head == 0) {
    if (P.splits == 1) {
      P.vis_stats[m * 3 + 0] = cnt;
      P.vis_stats[m * 3 + 1] = cnt ? first : -1;
      P.vis_stats[m * 3 + 2] = cnt ? last : -1;
    } else if (cnt) {
      atomicAdd(&P.vis_stats[m * 3 + 0], cnt);
      atomicMin(&P.vis_stats[m * 3 + 1], first);
      atomicMax(&P.vis_stats[m * 3 + 2], last);
    }
  }
}

__global__ void __launch_bounds__(THREADS, 1) latent_attn_tc_kernel(const __grid_constant__ AttnParams P) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  Bars* B = (Bars*)(smem + OFF_BAR);
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  const uint32_t rank = cluster_ctarank(), peer = rank ^ 1u;
  const int nch = rank == 0 ? 5 : 4;
  const int unit = blockIdx.x / 2;
  const int b = unit / P.tiles_per_block, qt = unit % P.tiles_per_block;
  const long row0 = ((long)b * P.tiles_per_block + qt) * QROWS;   // first Q_abs row of the tile

  if (tid == 0) {
    mbar_init(&B->q_full, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&B->kv_full[s], 1);
      mbar_init(&B->kv_empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&B->s_full[s], 1);
      mbar_init(&B->s_free[s], QROWS);
    }
    mbar_init(&B->p_full, QROWS);
    mbar_init(&B->o_done, 1);
    mbar_init(&B->x_full, 1);      // one arrival per tile from the peer
    mbar_init(&B->x_empty, 1);
    B->abort = 0;
    fence_mbar_init();
  }
  if (warp == 5) tmem_alloc(&B->tmem_slot, TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();          // the peer's barriers exist before anyone signals them
  tc_fence_after();
  const uint32_t tmem = B->tmem_slot;

  // key range of this tile: [j_lo, kvl) in 64-key tiles (identical in both CTAs)
  int kvl = P.kv_len[b];
  const int cap = P.max_pages * P.page_size;
  if (kvl < 0 || kvl > cap) {
    if (tid == 0 && rank == 0) set_status(P.status, MLA_DEV_BAD_LENGTH);
    kvl = max(0, min(kvl, cap));
  }
  const int W = P.window ? P.window[b] : 0;
  int j_lo = 0;
  if (W > 0) {
    const int t_first = (qt * QROWS) / P.H, t_last = (qt * QROWS + QROWS - 1) / P.H;
    int pmin = 0x7fffffff;
    for (int t = t_first; t <= t_last; ++t) pmin = min(pmin, P.positions[(long)b * P.T + t]);
    j_lo = max(0, pmin - W + 1) / KT * KT;
  }
  int nt = kvl > j_lo ? (kvl - j_lo + KT - 1) / KT : 0;
  {  // this split's share of the tiles
    const int tb = (int)((long)blockIdx.y * nt / P.splits);
    const int te = (int)((long)(blockIdx.y + 1) * nt / P.splits);
    j_lo += tb * KT;
    nt = te - tb;
  }

  if (warp == 4) {
    if (lane == 0) {
      // ---- TMA producer ----
      prefetch_tmap(&P.tmQ);
      prefetch_tmap(&P.tmKV);
      mbar_arrive_expect_tx(&B->q_full, nch * Q_CH_BYTES);
      for (int i = 0; i < nch; ++i)
        tma_load_3d(smem + OFF_Q + i * Q_CH_BYTES, &P.tmQ, &B->q_full, dim_chunk(rank, i) * DCH,
                    (int)row0, 0);
      const int R = P.seg_rows, past_end = P.num_pages * P.page_size;
      int issued = 0;
      // cache row of key j (beyond the cache when j is past kv_len or its page
      // is invalid: TMA then fills zeros)
      auto cache_row = [&](int j, bool report) {
        if (j >= kvl) return past_end;
        const int pg = P.block_table[(long)b * P.max_pages + j / P.page_size];
        if (pg >= 0 && pg < P.num_pages) return pg * P.page_size + j % P.page_size;
        if (report) set_status(P.status, MLA_DEV_BAD_PAGE);
        return past_end;
      };
      auto prefetch_tile = [&](int t) {
        if (t >= nt) return;
        for (int seg = 0; seg < KT / R; ++seg) {
          const int y = cache_row(j_lo + t * KT + seg * R, false);
          if (y == past_end) continue;
          for (int i = 0; i < nch; ++i) tma_prefetch_3d(&P.tmKV, dim_chunk(rank, i) * DCH, y, 0);
        }
      };
      prefetch_tile(0);
      prefetch_tile(1);
      for (int t = 0; t < nt; ++t) {
        const int s = t & 1;
        prefetch_tile(t + 2);
        if (!wait_local(B, &B->kv_empty[s], ((t >> 1) & 1) ^ 1, P.status)) break;
        const int j0 = j_lo + t * KT;
        uint8_t* stage = smem + OFF_KV + s * KV_STAGE_BYTES;
        mbar_arrive_expect_tx(&B->kv_full[s], nch * KV_CH_BYTES);
        for (int seg = 0; seg < KT / R; ++seg) {
          const int y = cache_row(j0 + seg * R, true);
          for (int i = 0; i < nch; ++i)
            tma_load_3d(stage + i * KV_CH_BYTES + seg * R * 128, &P.tmKV, &B->kv_full[s],
                        dim_chunk(rank, i) * DCH, y, 0);
        }
        issued = t + 1;
      }
      // every issued copy has landed before the CTA may exit
      mbar_wait(&B->q_full, 0, P.status);
      for (int t = max(0, issued - 2); t < issued; ++t)
        mbar_wait(&B->kv_full[t & 1], (t >> 1) & 1, P.status);
    }
  } else if (warp == 5) {
    if (lane == 0) {
      // ---- MMA issuer ----
      const uint32_t idesc_qk = idesc_f16(QROWS, KT, false);
      const uint32_t idesc_pv = idesc_f16_bmn(QROWS, 256, false);
      const bool have_q = wait_local(B, &B->q_full, 0, P.status);
      // S(t) = Q K(t)^T into score buffer t % 2 (its (t/2)-th use)
      auto issue_qk = [&](int t) -> bool {
        const int s = t & 1;
        if (!wait_local(B, &B->kv_full[s], (t >> 1) & 1, P.status)) return false;
        if (!wait_local(B, &B->s_free[s], ((t >> 1) & 1) ^ 1, P.status)) return false;
        tc_fence_after();
        const uint8_t* stage = smem + OFF_KV + s * KV_STAGE_BYTES;
        for (int i = 0; i < nch; ++i) {
          const uint64_t da = smem_desc_sw128(smem + OFF_Q + i * Q_CH_BYTES);
          const uint64_t db = smem_desc_sw128(stage + i * KV_CH_BYTES);
#pragma unroll
          for (int k = 0; k < DCH / 16; ++k)
            mma_f16(tmem + TM_S + 64 * s, da + 2 * k, db + 2 * k, idesc_qk, (i | k) != 0);
        }
        mma_commit(&B->s_full[s]);
        return true;
      };
      bool ok = have_q && (nt == 0 || issue_qk(0));
      for (int t = 0; t < nt && ok; ++t) {
        // the next tile's scores overlap this tile's softmax
        if (t + 1 < nt && !issue_qk(t + 1)) break;
        if (!wait_local(B, &B->p_full, t & 1, P.status)) break;
        tc_fence_after();
        const uint8_t* stage = smem + OFF_KV + (t & 1) * KV_STAGE_BYTES;
        const uint64_t dp = smem_desc_sw128(smem + OFF_P);
        const uint64_t dv = smem_desc_sw128_mn(stage, KV_CH_BYTES);
#pragma unroll
        for (int k = 0; k < KT / 16; ++k)   // 16 keys per MMA: 32 B along P rows, 16 V rows
          mma_f16(tmem + TM_O, dp + 2 * k, dv + (uint64_t)(16 * 128 / 16) * k, idesc_pv,
                  (t | k) != 0);
        mma_commit(&B->o_done);
        mma_commit(&B->kv_empty[t & 1]);
      }
    }
  } else {
    softmax_and_store(P, B, smem, tmem, rank, peer, b, qt, row0, kvl, W, j_lo, nt);
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();          // no CTA leaves while its peer may still signal it
  if (warp == 5) tmem_dealloc(tmem, TMEM_COLS);
}

}  // namespace
}  // namespace tc
}  // namespace mla

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
#include "gemm_tc.cuh"

namespace mla {
namespace tc {

mla_status_t latent_attention(cudaStream_t st, const mla_handle* h, const __nv_bfloat16* q_abs,
                              const __nv_bfloat16* cache, int num_pages,
                              const mla_attn_desc_t& d, const int32_t* positions, __half* o_lat,
                              float* part) {
  const Layout& l = h->lay;
  const int ps = h->cfg.page_size;
  if (l.rkv != 512 || l.dr != 64)
    return fail(MLA_ERR_UNSUPPORTED, "tcgen05 attention: needs kv_lora_rank 512, qk_rope_head_dim 64");
  if ((d.block_len * l.H) % QROWS)
    return fail(MLA_ERR_UNSUPPORTED, "tcgen05 attention: block_len * num_heads must be a multiple of 128");
  if (ps % 16 || (ps < KT && KT % ps) || (ps > KT && ps % KT))
    return fail(MLA_ERR_UNSUPPORTED, "tcgen05 attention: page_size must be 16, 32 or a multiple of 64");
  if (d.num_blocks <= 0) return MLA_OK;
  const long tokens = (long)d.num_blocks * d.block_len;
  const int splits = attn_splits(h, tokens);
  AttnParams P;
  const long rows = (long)d.num_blocks * d.block_len * l.H;
  if (!make_tmap_2d(&P.tmQ, false, q_abs, rows, l.L, l.L, QROWS) ||
      !make_tmap_2d(&P.tmKV, false, cache, (long)num_pages * ps, l.L, l.L, ps < KT ? ps : KT))
    return fail(MLA_ERR_CUDA, "tcgen05 attention: cuTensorMapEncodeTiled failed");
  P.block_table = d.block_table;
  P.kv_len = d.kv_len;
  P.window = d.window;
  P.q_visible = d.q_visible;
  P.positions = positions;
  P.vis_stats = d.vis_stats;
  P.o_lat = o_lat;
  P.status = h->status;
  P.max_pages = d.max_pages;
  P.num_pages = num_pages;
  P.page_size = ps;
  P.seg_rows = ps < KT ? ps : KT;
  P.T = d.block_len;
  P.H = l.H;
  P.tiles_per_block = d.block_len * l.H / QROWS;
  P.scale_log2 = h->scale * 1.4426950408889634f;
  P.splits = splits;
  P.rows = rows;
  P.o_part = part;
  P.lse_part = part + (size_t)splits * rows * 512;
  if (splits > 1 && d.vis_stats) init_vis_stats(st, d.vis_stats, tokens);
  static std::once_flag once;
  std::call_once(once, [] {
    cudaFuncSetAttribute(latent_attn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         SMEM_BYTES);
  });
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * d.num_blocks * P.tiles_per_block, splits, 1);
  cfg.blockDim = dim3(THREADS, 1, 1);
  cfg.dynamicSmemBytes = SMEM_BYTES;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, latent_attn_tc_kernel, P);
  if (e != cudaSuccess) return cuda_fail(e, "tcgen05 attention launch");
  if (splits > 1) merge_splits(st, P.o_part, P.lse_part, splits, rows, o_lat, d.vis_stats, l.H);
  return MLA_OK;
}

// Enough splits that the (block, 128-row) units fill every SM once, at most 8.
int attn_splits(const mla_handle* h, long tokens) {
  const long units = tokens * h->lay.H / QROWS;
  if (units <= 0) return 1;
  const long s = (h->num_sms + 2 * units - 1) / (2 * units);
  return (int)(s < 1 ? 1 : s > 8 ? 8 : s);
}

size_t attn_split_floats(const mla_handle* h, long tokens) {
  const int s = attn_splits(h, tokens);
  return s > 1 ? (size_t)s * tokens * h->lay.H * (512 + 1) : 0;
}

}  // namespace tc
}  // namespace mla
