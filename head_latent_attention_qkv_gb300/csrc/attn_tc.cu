// tcgen05 latent attention of the MLA draft layer ("MLA (Multi-Head Latent
// Attention)" blog, forward_mqa / decode_attention_fwd: one shared 576-wide
// latent KV head; queries absorbed into the latent space; output in the
// 512-wide latent value space).
//
// Work unit: one query block and 128 consecutive rows of Q_abs (rows are
// (token, head) pairs, token-major), handled by a cluster of two CTAs.  The
// 128 x 512 fp32 output accumulator does not fit one SM's tensor memory next
// to the score tiles, so CTA r keeps value columns [256r, 256r+256) in TMEM.
// The score reduction over the 576 latent dims is split between the pair:
// CTA 0 owns dims 0..255 and the rope dims 512..575, CTA 1 owns dims
// 256..511, which are also exactly the value dims each needs, so every cache
// byte is loaded once per pair.  Per 64-key tile t:
//   MMA warp      : S_r(t) = Q_r K_r(t)^T over its own dims into score buffer
//                   t % 2 (issued while the softmax still works on tile t-1)
//   exchange warps: as soon as S_r(t) lands, send it to the peer with
//                   asynchronous DSMEM stores that count their bytes on the
//                   peer's barrier (double-buffered, so the send overlaps the
//                   softmax of the previous tile)
//   softmax warps : add own and peer partial (same order in both CTAs, so
//                   both see identical scores), mask by logical position,
//                   online softmax in fp32 (exp2 domain; the TMEM accumulator
//                   is rescaled only when the running max grows by more than
//                   2^8), write P (bf16) into tensor memory, buffer t % 2
//   MMA warp      : O_r += P(t) V_r(t), P read from tensor memory, V read
//                   MN-major straight from the staged KV tile
// Warps 0-3 run the softmax and the epilogue (thread = accumulator row = TMEM
// lane), warps 4-7 the score exchange (same lanes), warp 8 streams Q and KV
// tiles with TMA, warp 9 owns TMEM and issues the MMAs.
#include "attn_tc.cuh"

#include <mutex>

#include "tc_ptx.cuh"

namespace mla {
namespace tc {
namespace {

constexpr int QROWS = 128, KT = 64, DCH = 64;    // query rows, keys per tile, dims per chunk
constexpr int THREADS = 320;
constexpr int MAX_CH = 5;                         // dim chunks held by CTA 0 (4 latent + rope)
constexpr int Q_CH_BYTES = QROWS * DCH * 2;       // 16 KiB
constexpr int KV_CH_BYTES = KT * DCH * 2;         // 8 KiB
constexpr int KV_STAGE_BYTES = MAX_CH * KV_CH_BYTES;
constexpr int X_BYTES = QROWS * KT * 4;           // one tile of peer partial scores
constexpr int OFF_Q = 0;
constexpr int OFF_KV = OFF_Q + MAX_CH * Q_CH_BYTES;
constexpr int OFF_X = OFF_KV + 2 * KV_STAGE_BYTES;
constexpr int OFF_BAR = OFF_X + 2 * X_BYTES;
constexpr int SMEM_BYTES = 1024 + OFF_BAR + 256;
// TMEM columns: O at 0..255, scores at 256 + 64 b, P (bf16 pairs) at 384 + 32 b
constexpr uint32_t TMEM_COLS = 512, TM_O = 0, TM_S = 256, TM_P = 384;
constexpr float RESCALE_LOG2 = 8.f;               // lazy rescale threshold (factor 256)

struct Bars {
  uint64_t q_full, kv_full[2], kv_empty[2], s_full[2], s_free[2], p_full, o_done[2];
  uint64_t x_full[2];    // peer's partial scores landed (expect-tx, 1 local arrival)
  uint64_t x_empty[2];   // peer has read the partial scores sent to it (4 warp arrivals)
  uint32_t tmem_slot;
  int abort;
};

__device__ __forceinline__ int dim_chunk(int rank, int i) {
  return rank == 0 ? (i < 4 ? i : 8) : 4 + i;    // global 64-dim chunk of local chunk i
}

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

// Warps 4-7: forward this CTA's partial scores of every tile to the peer.
__device__ __forceinline__ void exchange_scores(const AttnParams& P, Bars* B, uint8_t* smem,
                                                uint32_t tmem, uint32_t peer, int nt) {
  const int r = threadIdx.x - QROWS;                  // row / TMEM lane
  const uint32_t lane_base = (uint32_t)((r / 32) * 32) << 16;
  const uint32_t peer_x = mapa(smem_u32((float*)(smem + OFF_X) + r * KT), peer);
  const uint32_t peer_full[2] = {mapa(smem_u32(&B->x_full[0]), peer), mapa(smem_u32(&B->x_full[1]), peer)};
  for (int t = 0; t < nt; ++t) {
    const int buf = t & 1;
    const uint32_t ph = (t >> 1) & 1;
    if (!wait_local(B, &B->s_full[buf], ph, P.status)) break;
    tc_fence_after();
    float s[KT];
    tmem_ld32(tmem + TM_S + 64 * buf + lane_base, s);
    tmem_ld32(tmem + TM_S + 64 * buf + lane_base + 32, s + 32);
    tc_fence_before();
    mbar_arrive(&B->s_free[buf]);
    // the peer has read what was sent into this buffer two tiles ago
    if (!wait_peer(B, &B->x_empty[buf], ph ^ 1, P.status)) break;
    // 16-byte chunk c of a row sits at chunk c ^ (row % 8): the eight rows a
    // quarter-warp touches at once fall in distinct banks
#pragma unroll
    for (int c = 0; c < KT / 4; ++c)
      st_async_v4(peer_x + buf * X_BYTES + 16 * (c ^ (r & 7)), s[4 * c], s[4 * c + 1], s[4 * c + 2],
                  s[4 * c + 3], peer_full[buf]);
  }
}

// Warps 0-3: thread r owns accumulator row r (TMEM lane r) of the tile.
__device__ __forceinline__ void softmax_and_store(const AttnParams& P, Bars* B, uint8_t* smem,
                                                  uint32_t tmem, uint32_t rank, uint32_t peer,
                                                  int b, int qt, long row0, int kvl, int W,
                                                  int j_lo, int nt) {
  const int r = threadIdx.x, lane = r % 32;
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
  const float* xrow = (const float*)(smem + OFF_X) + r * KT;
  const uint32_t peer_empty[2] = {mapa(smem_u32(&B->x_empty[0]), peer), mapa(smem_u32(&B->x_empty[1]), peer)};
  float mrun = -INFINITY, lsum = 0.f;
  int cnt = 0, first = -1, last = -1;
  for (int t = 0; t < nt; ++t) {
    const int buf = t & 1;
    const uint32_t ph = (t >> 1) & 1;
    const int j0 = j_lo + t * KT;
    float s[KT];
    wait_local(B, &B->s_full[buf], ph, P.status);
    tc_fence_after();
    tmem_ld32(tmem + TM_S + 64 * buf + lane_base, s);
    tmem_ld32(tmem + TM_S + 64 * buf + lane_base + 32, s + 32);
    wait_peer(B, &B->x_full[buf], ph, P.status);
    // arm this buffer for tile t + 2 before the peer can be told it is free
    if (r == 0 && t + 2 < nt) mbar_arrive_expect_tx(&B->x_full[buf], X_BYTES);
    const float* x = xrow + buf * (X_BYTES / 4);
#pragma unroll
    for (int c = 0; c < KT / 4; ++c) {
      const float4 v = *reinterpret_cast<const float4*>(x + 4 * (c ^ (r & 7)));
      const float xs[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int u = 0; u < 4; ++u) s[4 * c + u] = rank == 0 ? s[4 * c + u] + xs[u] : xs[u] + s[4 * c + u];
    }
    tc_fence_before();
    mbar_arrive(&B->s_free[buf]);
    // mask by logical position (a warp whose rows all see the whole tile skips it)
    const int lo = max(vlo - j0, 0), hi = min(vhi - j0, KT);   // visible columns [lo, hi)
    if (hi > lo) {
      cnt += hi - lo;
      if (first < 0) first = j0 + lo;
      last = j0 + hi - 1;
    }
    float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
    if (__all_sync(0xffffffffu, lo == 0 && hi == KT)) {
#pragma unroll
      for (int i = 0; i < KT; ++i) mx4[i & 3] = fmaxf(mx4[i & 3], s[i]);
    } else {
#pragma unroll
      for (int i = 0; i < KT; ++i) {
        s[i] = (i >= lo && i < hi) ? s[i] : -INFINITY;
        mx4[i & 3] = fmaxf(mx4[i & 3], s[i]);
      }
    }
    // into the exp2 domain: the scale is positive, so it commutes with the max
    const float tmax = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3])) * P.scale_log2;
    const bool grow = tmax > mrun + RESCALE_LOG2;
    const float m_new = grow ? tmax : mrun;
    const float mref = m_new == -INFINITY ? 0.f : m_new;      // all masked so far: P = 0
    float ps4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int i = 0; i < KT; ++i) {
      s[i] = fast_exp2(fmaf(s[i], P.scale_log2, -mref));
      ps4[i & 3] += s[i];
    }
    const float psum = (ps4[0] + ps4[1]) + (ps4[2] + ps4[3]);
    const float alpha = (grow && mrun != -INFINITY) ? exp2f(mrun - m_new) : 1.f;
    if (t > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
      // every earlier P.V has finished before O is rescaled
      wait_local(B, &B->o_done[(t - 1) & 1], ((t - 1) >> 1) & 1, P.status);
      tc_fence_after();
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
    // P buffer `buf` was last read by P.V of tile t - 2
    if (t >= 2) {
      wait_local(B, &B->o_done[buf], ph ^ 1, P.status);
      tc_fence_after();
    }
    // value rows of keys past kv_len may hold anything: zero them (last tile)
    const bool tail = j0 + KT > kvl;
    if (tail) {
      uint8_t* stage = smem + OFF_KV + buf * KV_STAGE_BYTES;
      const int z0 = max(0, kvl - j0), pieces = (KT - z0) * 4 * 8;
      for (int idx = r; idx < pieces; idx += QROWS) {
        const int key = z0 + idx / 32, ch = (idx % 32) / 8, q = idx % 8;
        *reinterpret_cast<uint4*>(stage + ch * KV_CH_BYTES + key * 128 + q * 16) = make_uint4(0, 0, 0, 0);
      }
      fence_proxy_async_smem();
    }
    // P row in bf16 pairs: key 2c in the low half of column c
    float pw[KT / 2];
#pragma unroll
    for (int c = 0; c < KT / 2; ++c) {
      __nv_bfloat162 h2 = __floats2bfloat162_rn(s[2 * c], s[2 * c + 1]);
      pw[c] = *reinterpret_cast<float*>(&h2);
    }
    tmem_st32(tmem + TM_P + 32 * buf + lane_base, pw);
    tc_fence_before();
    mbar_arrive(&B->p_full);
    // this warp's reads of the exchange buffer are complete: the peer may
    // overwrite it (release orders those reads before the arrival)
    __syncwarp();
    if (lane == 0) mbar_arrive_remote(peer_empty[buf]);
  }
  // epilogue: O_r / l -> fp16 latent output columns [256 rank, 256 rank + 256)
  if (nt > 0) wait_local(B, &B->o_done[(nt - 1) & 1], ((nt - 1) >> 1) & 1, P.status);
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

  if (tid == 0) {
    mbar_init(&B->q_full, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&B->kv_full[s], 1);
      mbar_init(&B->kv_empty[s], 1);
      mbar_init(&B->s_full[s], 1);
      mbar_init(&B->s_free[s], 2 * QROWS);    // softmax and exchange threads
      mbar_init(&B->o_done[s], 1);
      mbar_init(&B->x_full[s], 1);
      mbar_init(&B->x_empty[s], QROWS / 32);  // one arrival per peer softmax warp
    }
    mbar_init(&B->p_full, QROWS);
    B->abort = 0;
    fence_mbar_init();
    // the first two score tiles from the peer are expected before it can send
    for (int s = 0; s < 2 && s < nt; ++s) mbar_arrive_expect_tx(&B->x_full[s], X_BYTES);
  }
  if (warp == 9) tmem_alloc(&B->tmem_slot, TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();          // the peer's barriers exist before anyone signals them
  tc_fence_after();
  const uint32_t tmem = B->tmem_slot;

  if (warp == 8) {
    if (lane == 0) {
      // ---- TMA producer ----
      prefetch_tmap(&P.tmQ);
      prefetch_tmap(&P.tmKV);
      mbar_arrive_expect_tx(&B->q_full, nch * Q_CH_BYTES);
      for (int i = 0; i < nch; ++i)
        tma_load_3d(smem + OFF_Q + i * Q_CH_BYTES, &P.tmQ, &B->q_full, dim_chunk(rank, i) * DCH,
                    (int)row0, 0);
      const int R = P.seg_rows, nseg = KT / R, past_end = P.num_pages * P.page_size;
      // cache row of key j (beyond the cache when j is past kv_len or its page
      // is invalid: TMA then fills zeros)
      auto cache_row = [&](int j) {
        if (j >= kvl) return past_end;
        const int pg = P.block_table[(long)b * P.max_pages + j / P.page_size];
        if (pg >= 0 && pg < P.num_pages) return pg * P.page_size + j % P.page_size;
        set_status(P.status, MLA_DEV_BAD_PAGE);
        return past_end;
      };
      // cache rows of tile t's segments (at most 4: page_size >= 16), looked
      // up and pulled into L2 two tiles ahead of the tile's load
      auto lookup = [&](int t, int* y) {
#pragma unroll
        for (int seg = 0; seg < 4; ++seg) {
          y[seg] = past_end;
          if (t < nt && seg < nseg) {
            y[seg] = cache_row(j_lo + t * KT + seg * R);
            if (y[seg] != past_end)
              for (int i = 0; i < nch; ++i) tma_prefetch_3d(&P.tmKV, dim_chunk(rank, i) * DCH, y[seg], 0);
          }
        }
      };
      int cur[4], nxt[4];
      lookup(0, cur);
      lookup(1, nxt);
      int issued = 0;
      for (int t = 0; t < nt; ++t) {
        const int s = t & 1;
        if (!wait_local(B, &B->kv_empty[s], ((t >> 1) & 1) ^ 1, P.status)) break;
        uint8_t* stage = smem + OFF_KV + s * KV_STAGE_BYTES;
        mbar_arrive_expect_tx(&B->kv_full[s], nch * KV_CH_BYTES);
#pragma unroll
        for (int seg = 0; seg < 4; ++seg)
          if (seg < nseg)
            for (int i = 0; i < nch; ++i)
              tma_load_3d(stage + i * KV_CH_BYTES + seg * R * 128, &P.tmKV, &B->kv_full[s],
                          dim_chunk(rank, i) * DCH, cur[seg], 0);
        issued = t + 1;
#pragma unroll
        for (int seg = 0; seg < 4; ++seg) cur[seg] = nxt[seg];
        lookup(t + 2, nxt);
      }
      // every issued copy has landed before the CTA may exit
      mbar_wait(&B->q_full, 0, P.status);
      for (int t = max(0, issued - 2); t < issued; ++t)
        mbar_wait(&B->kv_full[t & 1], (t >> 1) & 1, P.status);
    }
  } else if (warp == 9) {
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
        // the next tile's scores overlap this tile's exchange and softmax
        if (t + 1 < nt && !issue_qk(t + 1)) break;
        if (!wait_local(B, &B->p_full, t & 1, P.status)) break;
        tc_fence_after();
        const uint8_t* stage = smem + OFF_KV + (t & 1) * KV_STAGE_BYTES;
        const uint64_t dv = smem_desc_sw128_mn(stage, KV_CH_BYTES);
#pragma unroll
        for (int k = 0; k < KT / 16; ++k)   // 16 keys per MMA: 8 P columns, 16 V rows
          mma_f16_ts(tmem + TM_O, tmem + TM_P + 32 * (t & 1) + 8 * k,
                     dv + (uint64_t)(16 * 128 / 16) * k, idesc_pv, (t | k) != 0);
        mma_commit(&B->o_done[t & 1]);
        mma_commit(&B->kv_empty[t & 1]);
      }
    }
  } else if (warp >= 4) {
    exchange_scores(P, B, smem, tmem, peer, nt);
  } else {
    softmax_and_store(P, B, smem, tmem, rank, peer, b, qt, row0, kvl, W, j_lo, nt);
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();          // no CTA leaves while its peer may still signal it
  if (warp == 9) tmem_dealloc(tmem, TMEM_COLS);
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

// Clusters of the attention kernel resident on the GPU at once (queried once;
// also sets the kernel's shared-memory limit, so it runs before any launch).
static int attn_clusters_per_wave(const mla_handle* h) {
  static std::once_flag once;
  static int clusters = 0;
  std::call_once(once, [h] {
    cudaFuncSetAttribute(latent_attn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         SMEM_BYTES);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2, 1, 1);
    cfg.blockDim = dim3(THREADS, 1, 1);
    cfg.dynamicSmemBytes = SMEM_BYTES;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, latent_attn_tc_kernel, &cfg) != cudaSuccess || n <= 0) {
      (void)cudaGetLastError();
      n = h->num_sms / 2;
    }
    clusters = n;
  });
  return clusters;
}

// When the (block, 128-row) units leave part of the GPU idle, split each
// unit's key range so that the clusters fill one wave (at most 8 parts); a
// split that would add a partial wave only lengthens the kernel.
int attn_splits(const mla_handle* h, long tokens) {
  const long units = tokens * h->lay.H / QROWS;
  const long wave = attn_clusters_per_wave(h);
  if (units <= 0 || units >= wave) return 1;
  const long s = wave / units;
  return (int)(s < 1 ? 1 : s > 8 ? 8 : s);
}

size_t attn_split_floats(const mla_handle* h, long tokens) {
  const int s = attn_splits(h, tokens);
  return s > 1 ? (size_t)s * tokens * h->lay.H * (512 + 1) : 0;
}

}  // namespace tc
}  // namespace mla
