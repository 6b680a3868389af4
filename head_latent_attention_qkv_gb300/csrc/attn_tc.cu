// tcgen05 latent attention of the MLA draft layer ("MLA (Multi-Head Latent
// Attention)" blog, forward_mqa / decode_attention_fwd: one shared 576-wide
// latent KV head; queries absorbed into the latent space; output in the
// 512-wide latent value space).
//
// Work unit: one query block and 128 consecutive rows of Q_abs (rows are
// (token, head) pairs, token-major; a block's last tile is padded when
// block_len x heads is not a multiple of 128: its extra rows are fully masked
// and written nowhere), handled by a cluster of two CTAs, one per half of the
// 512 latent value dims.  A 128 x 512 fp32 accumulator would fill all of an
// SM's tensor memory, so each CTA keeps O for its 256 value dims and computes
// the full 576-wide scores itself (QK^T is repeated by the two halves).  Keys
// go in tiles of 128 (one MMA costs about the same for any N up to 128, so
// narrower score tiles waste the tensor pipe).
//
// The cache entries are keys and values at once: the four 64-dim chunks of a
// tile that hold this CTA's value half ("value chunks") arrive in one copy
// into the V buffer and serve both as B operand of QK^T (K-major) and of P V
// (MN-major); the other five chunks of the tile stream through a 5-slot ring.
// Each tile thus reads its 128 cache rows once per CTA; the ring holds a
// whole tile's five chunks, refilled as soon as the tile's MMAs are done with
// it, so that the next tile's chunks are resident long before they are read
// (one barrier for the ring: each mbarrier check costs the single MMA-issuing
// thread about 200 cycles, each tcgen05.mma about 110).
//
// Tensor memory (512 columns): O at 0..255, S (fp32, 128 keys) at 256..383,
// P (bf16 pairs, written over the first half of S once the softmax has read
// it) at 256..319, Q_abs dims 0..255 (bf16 pairs, A operand of four score
// chunks) at 384..511.
// Shared memory: Q_abs dims 256..575 (five chunks, one TMA copy), the V
// buffer (four value chunks of one tile, one copy), the 5-slot ring.
//
// Per tile t the tensor pipe runs S(t) over the ring chunks, then over the
// value chunks, then (once the softmax has written P(t)) O += P(t) V(t);
// S(t + 1)'s ring chunks are already resident by then, and V(t + 1) is
// copied while they are multiplied.
//   MMA warp     : S(t) = Q K(t)^T (36 MMAs, N = 128); O += P(t) V(t) (8 MMAs,
//                  N = 256, P read from tensor memory)
//   softmax warps (0-3 and 8-11): two threads per row r (TMEM lane r), each
//                  on 64 of the tile's keys and 128 of the value columns,
//                  exchanging the half maxima through shared memory: mask by
//                  logical position (one visible interval per row), online
//                  softmax in fp32 in the exp2 domain (O rescaled in tensor
//                  memory only when the running max grows by more than 2^8),
//                  P -> bf16 (one thread per row: ≈1.7 k of ≈6.2 k cycles per
//                  tile, with the tensor pipe waiting)
//   TMA warps    : warp 4 the page rows of the key range (once), Q, V(t);
//                  warps 6 and 7 the ring chunks (copies of different warps
//                  proceed side by side)
// The key range of a unit may be split (grid y) when units alone do not fill
// the GPU (the blog's forward_mqa num_kv_splits); the pairs of one unit then form
// one cluster of 2 x splits CTAs.  Every CTA stages its normalised partial
// output, its log2-sum-exp and visibility counts in its own shared memory
// (over the Q and V buffers, free after the last P V); after a cluster
// barrier split s combines rows [128 s / splits, 128 (s + 1) / splits) of its
// value half from all splits, in split order, by log-sum-exp (the blog's
// forward_mha merge_attn_states) and writes them as fp16 whole rows.
#include "attn_tc.cuh"

#include <mutex>

#include "tc_ptx.cuh"

namespace mla {
namespace tc {
namespace {

constexpr int QROWS = 128, KT = 128, DCH = 64, NCH = 9;  // rows, keys per tile, dims per chunk
constexpr int NQT = 4;                                    // Q chunks held in tensor memory
constexpr int NQS = NCH - NQT;                            // Q chunks held in shared memory
constexpr int NVC = 4;                                    // value chunks of this CTA's half
constexpr int NRC = NCH - NVC;                            // ring chunks per tile
constexpr int RSLOTS = NRC;                               // ring slot i holds ring chunk i
constexpr int THREADS = 384;                              // softmax x4, TMA, MMA, TMA x2, softmax x4
constexpr int Q_CH_BYTES = QROWS * DCH * 2;               // 16 KiB
constexpr int KV_CH_BYTES = KT * DCH * 2;                 // 16 KiB
constexpr int OFF_Q = 0;
constexpr int OFF_V = OFF_Q + NQS * Q_CH_BYTES;
constexpr int OFF_K = OFF_V + NVC * KV_CH_BYTES;
constexpr int OFF_BAR = OFF_K + RSLOTS * KV_CH_BYTES;
constexpr int OFF_PG = OFF_BAR + 256;                     // cache row of each page of the key range
constexpr int MAX_PG = 176;                               // pages held there (else looked up per load)
constexpr int OFF_XM = OFF_PG + MAX_PG * 4;               // [128] a row's half maximum (or sum)
constexpr int SMEM_BYTES = 1024 + OFF_XM + QROWS * 4 * 2;
constexpr uint32_t TMEM_COLS = 512, TM_O = 0, TM_S = 256, TM_P = 256, TM_Q = 384;
constexpr float RESCALE_LOG2 = 8.f;                       // lazy rescale threshold (factor 256)
constexpr int MAX_SPLITS = 4;                             // clusters of at most 8 CTAs
constexpr float kLn2 = 0.6931471805599453f;
// epilogue staging (over the Q and V buffers): fp32 rows of this CTA's 256
// value dims (pitch 260 floats: conflict-free 16-byte row-per-thread
// stores), then the rows' log2-sum-exp and visibility counts
constexpr int STG_PITCH = 256 + 4;
constexpr int OFF_STG = 0;
constexpr int OFF_LSE = OFF_STG + QROWS * STG_PITCH * 4;
constexpr int OFF_VS = OFF_LSE + QROWS * 4;
static_assert(OFF_VS + QROWS * 12 <= OFF_K, "staging fits over Q and V");

// Cache chunk held by ring slot i for value half h: the chunks outside
// [4h, 4h + 4), in increasing order.
__device__ __forceinline__ int ring_chunk(int i, int half) {
  return half == 0 ? NVC + i : (i < NVC ? i : NCH - 1);
}

struct Bars {
  uint64_t q_full;                    // Q chunks in shared memory (TMA)
  uint64_t q_tmem;                    // Q chunks in tensor memory (128 arrivals)
  uint64_t r_full;                    // the tile's ring chunks landed (phase t; two producers)
  uint64_t r_empty;                   // the MMAs reading the ring are done (phase t)
  uint64_t v_full;                    // V(t) landed (phase t)
  uint64_t s_full;                    // S(t) complete (phase t); also P(t - 1) V(t - 1)
  uint64_t p_full;                    // P(t) written (phase t)
  uint64_t o_done;                    // P(t) V(t) complete (phase t): the V buffer is free
  uint64_t drain;                     // every MMA of the CTA complete
  uint32_t tmem_slot;
  int abort;
};
static_assert(sizeof(Bars) <= 256, "barrier block");
static_assert(SMEM_BYTES <= 232448, "shared memory");

// Bounded wait that gives up at once after any earlier timeout of this CTA.
__device__ __forceinline__ bool wait_bar(Bars* B, uint64_t* bar, uint32_t parity, uint32_t* st) {
  if (*(volatile int*)&B->abort) return false;
  if (mbar_wait(bar, parity, st)) return true;
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

__device__ __forceinline__ void softmax_sync() { asm volatile("bar.sync 3, 256;" ::: "memory"); }

// Warps 0-3 and 8-11: the two threads of row r (TMEM lane r; warps w and
// w + 8 share the lane sub-partition) own key columns [64 kh, 64 kh + 64) of
// each score tile and value columns [128 kh, 128 kh + 128) of O.  They
// exchange their half's maximum each tile (and their half's sum at the end)
// through shared memory.
__device__ __forceinline__ void softmax_and_stage(const AttnParams& P, Bars* B, uint8_t* smem,
                                                  uint32_t tmem, int b, int qt, long row0, int kvl,
                                                  int W, int j_lo, int nt) {
  const int r = threadIdx.x & (QROWS - 1), kh = threadIdx.x >= 256 ? 1 : 0;
  constexpr int KH = KT / 2;                                   // score columns per thread
  const uint32_t lane_base = (uint32_t)((r / 32) * 32) << 16;
  float* xm = (float*)(smem + OFF_XM);                         // [2][128]
  const int row_in_block = qt * QROWS + r;
  // rows past the block's T x H (a partial last tile) are padding: fully masked
  const bool live = row_in_block < P.T * P.H;
  const long m = (long)b * P.T + (live ? row_in_block / P.H : 0);
  const int p = P.positions[m];
  const bool qv = live && (P.q_visible ? P.q_visible[m] != 0 : true);
  // the keys this query sees form one interval [vlo, vhi): j < kv_len and, for
  // a sliding window, p - j < W; a fully masked query sees none
  const int vlo = W > 0 ? max(0, p - W + 1) : 0;
  const int vhi = qv ? kvl : 0;
  float mrun = -INFINITY, lsum = 0.f;
  int cnt = 0, first = -1, last = -1;
  if (nt > 0) {
    // Q_abs dims 0..255 of this row -> tensor memory (bf16 pairs, low half = even dim)
    const uint4* src = reinterpret_cast<const uint4*>(P.q_abs + (row0 + r) * 576);
#pragma unroll 1
    for (int c = kh * (NQT / 2); c < (kh + 1) * (NQT / 2); ++c) {
      uint32_t w[32];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const uint4 v = live ? __ldg(src + c * 8 + i) : make_uint4(0, 0, 0, 0);
        w[4 * i] = v.x; w[4 * i + 1] = v.y; w[4 * i + 2] = v.z; w[4 * i + 3] = v.w;
      }
      tmem_st32_u(tmem + TM_Q + 32 * c + lane_base, w);
    }
    tc_fence_before();
    mbar_arrive(&B->q_tmem);
  }
  for (int t = 0; t < nt; ++t) {
    const uint32_t ph = t & 1;
    const int j0 = j_lo + t * KT;
    float s[KH];
    // S(t) complete (and, the MMAs completing in order, P(t - 1) V(t - 1))
    wait_bar(B, &B->s_full, ph, P.status);
    tc_fence_after();
#pragma unroll
    for (int c = 0; c < KH; c += 32) tmem_ld32_nowait(tmem + TM_S + KH * kh + c + lane_base, s + c);
    tmem_ld_wait();
#pragma unroll
    for (int c = 0; c < KH; c += 32) tmem_reg_fence32(s + c);
    // mask by logical position (a warp whose rows all see its half of the tile skips it)
    const int lo = max(vlo - j0, 0), hi = min(vhi - j0, KT);   // visible columns [lo, hi)
    if (hi > lo) {
      cnt += hi - lo;
      if (first < 0) first = j0 + lo;
      last = j0 + hi - 1;
    }
    const int lo_h = lo - KH * kh, hi_h = hi - KH * kh;          // the same, in this half
    float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
    if (__all_sync(0xffffffffu, lo_h <= 0 && hi_h >= KH)) {
#pragma unroll
      for (int i = 0; i < KH; ++i) mx4[i & 3] = fmaxf(mx4[i & 3], s[i]);
    } else {
#pragma unroll
      for (int i = 0; i < KH; ++i) {
        s[i] = (i >= lo_h && i < hi_h) ? s[i] : -INFINITY;
        mx4[i & 3] = fmaxf(mx4[i & 3], s[i]);
      }
    }
    // the row's maximum from both halves; into the exp2 domain (the scale is
    // positive, so it commutes with the max)
    const float hmax = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3]));
    xm[kh * QROWS + r] = hmax;
    softmax_sync();
    const float tmax = fmaxf(hmax, xm[(1 - kh) * QROWS + r]) * P.scale_log2;
    softmax_sync();                                            // both halves read before the next write
    const bool grow = tmax > mrun + RESCALE_LOG2;
    const float m_new = grow ? tmax : mrun;
    const float mref = m_new == -INFINITY ? 0.f : m_new;      // all masked so far: P = 0
    float ps4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int i = 0; i < KH; ++i) {
      s[i] = fast_exp2(fmaf(s[i], P.scale_log2, -mref));
      ps4[i & 3] += s[i];
    }
    const float psum = (ps4[0] + ps4[1]) + (ps4[2] + ps4[3]);
    const float alpha = (grow && mrun != -INFINITY) ? exp2f(mrun - m_new) : 1.f;
    // P(t - 1) V(t - 1) has completed (before S(t)): O may be rescaled
    if (t > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll 1
      for (int c = 128 * kh; c < 128 * kh + 128; c += 32) {
        float o[32];
        tmem_ld32(tmem + TM_O + lane_base + c, o);
#pragma unroll
        for (int i = 0; i < 32; ++i) o[i] *= alpha;
        tmem_st32(tmem + TM_O + lane_base + c, o);
      }
    }
    lsum = lsum * alpha + psum;
    mrun = m_new;
    // value rows of keys past kv_len may hold anything: S(t) is done with the
    // V buffer, zero those rows before P V reads them (last tile only)
    if (j0 + KT > kvl) {
      wait_bar(B, &B->v_full, ph, P.status);
      uint8_t* vbase = smem + OFF_V;
      const int z0 = max(0, kvl - j0), pieces = (KT - z0) * NVC * 8;
      for (int idx = r + QROWS * kh; idx < pieces; idx += 2 * QROWS) {
        const int key = z0 + idx / 32, ch = (idx % 32) / 8, q = idx % 8;
        *reinterpret_cast<uint4*>(vbase + ch * KV_CH_BYTES + key * 128 + q * 16) = make_uint4(0, 0, 0, 0);
      }
      fence_proxy_async_smem();
    }
    // P row in bf16 pairs over S (this thread has read its lane): key 2c in
    // the low half of column c
    {
      uint32_t pw[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        __nv_bfloat162 h2 = __floats2bfloat162_rn(s[2 * i], s[2 * i + 1]);
        pw[i] = *reinterpret_cast<uint32_t*>(&h2);
      }
      tmem_st32_u(tmem + TM_P + 32 * kh + lane_base, pw);
    }
    tc_fence_before();
    mbar_arrive(&B->p_full);
  }
  // stage this split's partial: O / l in fp32, log2-sum-exp, visibility counts
  // (the row sum from both halves)
  xm[kh * QROWS + r] = lsum;
  softmax_sync();
  lsum += xm[(1 - kh) * QROWS + r];
  if (nt > 0) wait_bar(B, &B->o_done, (nt - 1) & 1, P.status);
  tc_fence_after();
  const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
  const bool any = nt > 0 && lsum > 0.f;
  float* prow = (float*)(smem + OFF_STG) + r * STG_PITCH;
#pragma unroll 1
  for (int c = 128 * kh; c < 128 * kh + 128; c += 32) {
    float o[32];
    if (nt > 0) tmem_ld32(tmem + TM_O + lane_base + c, o);
#pragma unroll
    for (int i = 0; i < 32; i += 4)
      *reinterpret_cast<float4*>(prow + c + i) =
          any ? make_float4(o[i] * inv, o[i + 1] * inv, o[i + 2] * inv, o[i + 3] * inv)
              : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  if (kh == 0) {
    ((float*)(smem + OFF_LSE))[r] = any ? mrun + log2f(lsum) : -INFINITY;
    int* vs = (int*)(smem + OFF_VS) + 3 * r;
    vs[0] = cnt;
    vs[1] = first;
    vs[2] = last;
  }
}

__device__ __forceinline__ int ld_cluster_s32(uint32_t addr) {
  int v;
  asm volatile("ld.shared::cluster.s32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ float4 ld_cluster_v4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(addr) : "memory");
  return v;
}

// All warps, after every split has staged: rows [128 split / S, 128 (split +
// 1) / S) of value half `half`.  The merged row is sum_s w_s o_s / sum_s w_s,
// w_s = 2^(lse_s - max lse), added in split order; a row no split saw stays
// exactly zero.  Lane l writes value dims 8 l .. 8 l + 7 (a warp per row: one
// 512-byte write).  CTA (half h, split s) is cluster rank h + 2 s.
__device__ __forceinline__ void reduce_splits(const AttnParams& P, uint8_t* smem, int half,
                                              int split, int b, int qt, long row0) {
  const int S = P.splits;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int r_lo = split * QROWS / S, r_hi = (split + 1) * QROWS / S;
  const uint32_t stg = smem_u32(smem + OFF_STG), lse_a = smem_u32(smem + OFF_LSE),
                 vs_a = smem_u32(smem + OFF_VS);
  if (S == 1) {
    // one split: this CTA's own rows, normalised already
    const float* lse = (const float*)(smem + OFF_LSE);
    const int* vs = (const int*)(smem + OFF_VS);
    const int rows = min(QROWS, P.T * P.H - qt * QROWS);   // live rows of this tile
    for (int r = warp; r < rows; r += THREADS / 32) {
      const float4* src = (const float4*)(smem + OFF_STG + (r * STG_PITCH + 8 * lane) * 4);
      const float4 a = src[0], c = src[1];
      const bool any = lse[r] != -INFINITY;
      __half2 h2[4] = {__floats2half2_rn(any ? a.x : 0.f, any ? a.y : 0.f),
                       __floats2half2_rn(any ? a.z : 0.f, any ? a.w : 0.f),
                       __floats2half2_rn(any ? c.x : 0.f, any ? c.y : 0.f),
                       __floats2half2_rn(any ? c.z : 0.f, any ? c.w : 0.f)};
      *reinterpret_cast<uint4*>(P.o_lat + (row0 + r) * 512 + half * 256 + 8 * lane) =
          *reinterpret_cast<uint4*>(h2);
      const int row_in_block = qt * QROWS + r;
      if (P.lse && half == 0 && lane == 0) P.lse[row0 + r] = any ? lse[r] * kLn2 : -INFINITY;
      if (P.vis_stats && half == 0 && row_in_block % P.H == 0 && lane == 0) {
        const long m = (long)b * P.T + row_in_block / P.H;
        const int cnt = vs[3 * r];
        P.vis_stats[m * 3 + 0] = cnt;
        P.vis_stats[m * 3 + 1] = cnt ? vs[3 * r + 1] : -1;
        P.vis_stats[m * 3 + 2] = cnt ? vs[3 * r + 2] : -1;
      }
    }
    return;
  }
  const int rows = min(r_hi, P.T * P.H - qt * QROWS);   // live rows of this tile
  for (int r = r_lo + warp; r < rows; r += THREADS / 32) {
    const uint32_t off = stg + (uint32_t)(r * STG_PITCH + 8 * lane) * 4;
    float lse[MAX_SPLITS];
    float4 v[MAX_SPLITS][2];
#pragma unroll
    for (int s = 0; s < MAX_SPLITS; ++s) {
      if (s < S) {
        const uint32_t rank = (uint32_t)(half + 2 * s);
        lse[s] = ld_cluster_f32(mapa(lse_a + 4 * r, rank));
        v[s][0] = ld_cluster_v4(mapa(off, rank));
        v[s][1] = ld_cluster_v4(mapa(off + 16, rank));
      }
    }
    float mx = -INFINITY;
#pragma unroll
    for (int s = 0; s < MAX_SPLITS; ++s)
      if (s < S) mx = fmaxf(mx, lse[s]);
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f}, den = 0.f;
#pragma unroll
    for (int s = 0; s < MAX_SPLITS; ++s) {
      if (s < S) {
        const float w = mx == -INFINITY ? 0.f : exp2f(lse[s] - mx);
        den += w;
        acc[0] += w * v[s][0].x; acc[1] += w * v[s][0].y; acc[2] += w * v[s][0].z; acc[3] += w * v[s][0].w;
        acc[4] += w * v[s][1].x; acc[5] += w * v[s][1].y; acc[6] += w * v[s][1].z; acc[7] += w * v[s][1].w;
      }
    }
    const float inv = den > 0.f ? 1.f / den : 0.f;
    if (P.lse && half == 0 && lane == 0)
      P.lse[row0 + r] = den > 0.f ? (mx + log2f(den)) * kLn2 : -INFINITY;
    __half2 h2[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) h2[u] = __floats2half2_rn(acc[2 * u] * inv, acc[2 * u + 1] * inv);
    *reinterpret_cast<uint4*>(P.o_lat + (row0 + r) * 512 + half * 256 + 8 * lane) =
        *reinterpret_cast<uint4*>(h2);
    // visibility statistics of the row's token (from the head-0 row, value half 0)
    const int row_in_block = qt * QROWS + r;
    if (P.vis_stats && half == 0 && row_in_block % P.H == 0 && lane == 0) {
      int cnt = 0, first = -1, last = -1;
      for (int s = 0; s < S; ++s) {
        const uint32_t a = mapa(vs_a + 12 * r, (uint32_t)(2 * s));
        const int c = ld_cluster_s32(a), f = ld_cluster_s32(a + 4), l = ld_cluster_s32(a + 8);
        if (c) {
          first = cnt ? min(first, f) : f;
          last = max(last, l);
          cnt += c;
        }
      }
      const long m = (long)b * P.T + row_in_block / P.H;
      P.vis_stats[m * 3 + 0] = cnt;
      P.vis_stats[m * 3 + 1] = cnt ? first : -1;
      P.vis_stats[m * 3 + 2] = cnt ? last : -1;
    }
  }
}

__global__ void __launch_bounds__(THREADS, 1) latent_attn_tc_kernel(const __grid_constant__ AttnParams P) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  Bars* B = (Bars*)(smem + OFF_BAR);
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  const int rank = (int)cluster_ctarank();             // half + 2 * split
  const int half = rank & 1, split = rank >> 1;         // split == blockIdx.y
  const int unit = blockIdx.x >> 1;
  const int b = unit / P.tiles_per_block, qt = unit % P.tiles_per_block;
  const long row0 = (long)b * P.T * P.H + (long)qt * QROWS;       // first Q_abs row of the unit

  // key range of this unit: [j_lo, kvl) in 128-key tiles (identical in both halves)
  int kvl = P.kv_len[b];
  const int cap = P.max_pages * P.page_size;
  if (kvl < 0 || kvl > cap) {
    if (tid == 0 && half == 0) set_status(P.status, MLA_DEV_BAD_LENGTH);
    kvl = max(0, min(kvl, cap));
  }
  const int W = P.window ? P.window[b] : 0;
  if (W < 0) {                 // rejected: the block's rows see no key (exact zeros)
    if (tid == 0 && half == 0 && blockIdx.y == 0) set_status(P.status, MLA_DEV_BAD_WINDOW);
    kvl = 0;
  }
  int j_lo = 0;
  if (W > 0) {
    const int t_first = (qt * QROWS) / P.H, t_last = min(P.T - 1, (qt * QROWS + QROWS - 1) / P.H);
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
    mbar_init(&B->q_tmem, 2 * QROWS);
    mbar_init(&B->r_full, 2);
    mbar_init(&B->r_empty, 1);
    mbar_init(&B->v_full, 1);
    mbar_init(&B->s_full, 1);
    mbar_init(&B->p_full, 2 * QROWS);
    mbar_init(&B->o_done, 1);
    mbar_init(&B->drain, 1);
    B->abort = 0;
    fence_mbar_init();
  }
  if (warp == 5) tmem_alloc(&B->tmem_slot, TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();          // every CTA of the cluster is resident before any DSMEM access
  tc_fence_after();
  const uint32_t tmem = B->tmem_slot;
  if (tid == 0) pdl_trigger();
  pdl_wait();                  // Q_abs and the block's own latents come from the kernels before

  if (warp == 4 || warp == 6 || warp == 7) {
    // the cache row of every page this CTA reads, looked up once by warp 4
    // (past_end for a page the table marks invalid: TMA then reads zeros)
    const int ps = P.page_size, past_end = P.num_pages * ps;
    const int p0 = j_lo / ps;
    const int npg = nt > 0 ? (min(kvl, j_lo + nt * KT) - 1) / ps - p0 + 1 : 0;
    int* pg_row = (int*)(smem + OFF_PG);
    const bool table = npg <= MAX_PG;
    if (warp == 4 && table) {
      for (int i = lane; i < npg; i += 32) {
        const int pg = P.block_table[(long)b * P.max_pages + p0 + i];
        const bool okp = pg >= 0 && pg < P.num_pages;
        if (!okp) set_status(P.status, MLA_DEV_BAD_PAGE);
        pg_row[i] = okp ? pg * ps : past_end;
      }
    }
    // the three producer warps (4, 6, 7) see the table before any copy
    asm volatile("bar.sync 1, 96;" ::: "memory");
    if (lane == 0 && nt > 0) {
      const int R = P.seg_rows, nseg = KT / R;
      // cache row of key j (beyond the cache when j is past kv_len or its page
      // is invalid: TMA then fills zeros)
      auto cache_row = [&](int j) {
        if (j >= kvl) return past_end;
        int base;
        if (table) {
          base = pg_row[j / ps - p0];
        } else {
          const int pg = P.block_table[(long)b * P.max_pages + j / ps];
          base = pg >= 0 && pg < P.num_pages ? pg * ps : past_end;
          if (base == past_end) set_status(P.status, MLA_DEV_BAD_PAGE);
        }
        return base == past_end ? past_end : base + j % ps;
      };
      // rows of tile t: one run of KT contiguous cache rows (first row
      // returned) or -1 when its segments must be copied one by one; rows past
      // kv_len inside the run are read but masked (scores) and zeroed (values)
      auto tile_run = [&](int t) {
        const int j0 = j_lo + t * KT;
        const int y0 = cache_row(j0);
        if (y0 == past_end || y0 + KT > past_end) return -1;
        for (int seg = 1; seg < nseg; ++seg) {
          const int j = j0 + seg * R;
          if (j < kvl && cache_row(j) != y0 + seg * R) return -1;
        }
        return y0;
      };
      if (warp == 4) {
        // ---- Q once, then V(t) for every tile, each as soon as P(t - 1) V(t - 1)
        // has freed the buffer ----
        prefetch_tmap(&P.tmQ);
        prefetch_tmap(&P.tmV);
        prefetch_tmap(&P.tmKs);
        mbar_arrive_expect_tx(&B->q_full, NQS * Q_CH_BYTES);
        tma_load_3d(smem + OFF_Q, &P.tmQ, &B->q_full, 0, (int)row0, NQT);
        for (int t = 0; t < nt; ++t) {
          if (t >= 1 && !wait_bar(B, &B->o_done, (t - 1) & 1, P.status)) break;
          mbar_arrive_expect_tx(&B->v_full, NVC * KV_CH_BYTES);
          const int y0 = tile_run(t);
          if (y0 >= 0) {
            tma_load_3d(smem + OFF_V, &P.tmV, &B->v_full, 0, y0, NVC * half);
          } else {
            for (int i = 0; i < NVC; ++i)
              for (int seg = 0; seg < nseg; ++seg)
                tma_load_3d(smem + OFF_V + i * KV_CH_BYTES + seg * R * 128, &P.tmKs, &B->v_full,
                            (NVC * half + i) * DCH, cache_row(j_lo + t * KT + seg * R), 0);
          }
        }
        // every copy into this CTA has landed before it may exit
        mbar_wait(&B->q_full, 0, P.status);
        mbar_wait(&B->v_full, (nt - 1) & 1, P.status);
      } else {
        // ---- ring: warp 6 refills slots 0, 2, 4, warp 7 slots 1, 3, each
        // once the MMAs of the previous tile are done with the whole ring ----
        prefetch_tmap(&P.tmK);
        prefetch_tmap(&P.tmKs);
        const int s0 = warp - 6;
        bool ok = true;
        for (int t = 0; t < nt && ok; ++t) {
          const int y0 = tile_run(t);
          if (!wait_bar(B, &B->r_empty, (t & 1) ^ 1, P.status)) { ok = false; break; }
          mbar_arrive_expect_tx(&B->r_full, (s0 == 0 ? 3 : 2) * KV_CH_BYTES);
          for (int i = s0; i < RSLOTS; i += 2) {
            uint8_t* dst = smem + OFF_K + i * KV_CH_BYTES;
            const int c = ring_chunk(i, half);
            if (y0 >= 0) {
              tma_load_3d(dst, &P.tmK, &B->r_full, c * DCH, y0, 0);
            } else {
              for (int seg = 0; seg < nseg; ++seg)
                tma_load_3d(dst + seg * R * 128, &P.tmKs, &B->r_full, c * DCH,
                            cache_row(j_lo + t * KT + seg * R), 0);
            }
          }
        }
        mbar_wait(&B->r_full, (nt - 1) & 1, P.status);
      }
    }
  } else if (warp == 5) {
    if (lane == 0 && nt > 0) {
      // ---- MMA issuer ----
      const uint32_t idesc_qk = idesc_f16(QROWS, KT, false);
      const uint32_t idesc_pv = idesc_f16_bmn(QROWS, 256, false);
      bool ok = wait_bar(B, &B->q_full, 0, P.status) && wait_bar(B, &B->q_tmem, 0, P.status);
      // S += Q[:, chunk] K(chunk)^T over the 576 dims, fully unrolled from
      // descriptors computed once (the issuing thread's rate is set by the
      // instructions between its MMAs): A is Q chunk qc in tensor memory
      // (dims 0..255) or smem Q chunk qs (dims 256..575), B the 128 keys'
      // chunk (K-major).  Half 0 reads Q chunks 4..8 with its ring and 0..3
      // with its value chunks; half 1 Q chunks 0..3 and 8 with its ring and
      // 4..7 with its value chunks.
      const uint64_t dK = smem_desc_sw128(smem + OFF_K), dVk = smem_desc_sw128(smem + OFF_V);
      const uint64_t dQs = smem_desc_sw128(smem + OFF_Q);
      const uint64_t dv = smem_desc_sw128_mn(smem + OFF_V, KV_CH_BYTES);
      constexpr uint32_t U_CH = KV_CH_BYTES / 16, U_Q = Q_CH_BYTES / 16, U_KSTEP = 16 * 128 / 16;
      const uint32_t tS = tmem + TM_S, tQ = tmem + TM_Q, tO = tmem + TM_O, tP = tmem + TM_P;
      auto qk_tm = [&](int qc, uint64_t db, uint32_t acc0) {
        mma_f16_ts(tS, tQ + 32 * qc, db, idesc_qk, acc0);
        mma_f16_ts(tS, tQ + 32 * qc + 8, db + 2, idesc_qk, 1u);
        mma_f16_ts(tS, tQ + 32 * qc + 16, db + 4, idesc_qk, 1u);
        mma_f16_ts(tS, tQ + 32 * qc + 24, db + 6, idesc_qk, 1u);
      };
      auto qk_sm = [&](int qs, uint64_t db, uint32_t acc0) {
        const uint64_t da = dQs + qs * U_Q;
        mma_f16(tS, da, db, idesc_qk, acc0);
        mma_f16(tS, da + 2, db + 2, idesc_qk, 1u);
        mma_f16(tS, da + 4, db + 4, idesc_qk, 1u);
        mma_f16(tS, da + 6, db + 6, idesc_qk, 1u);
      };
      for (int t = 0; t < nt && ok; ++t) {
        const uint32_t ph = t & 1;
        // S(t): the ring chunks, then the value chunks (P(t - 1) V(t - 1),
        // issued before, has read P out of these columns: same issuing
        // thread, executed in order)
        if (!(ok = wait_bar(B, &B->r_full, ph, P.status))) break;
        tc_fence_after();
        if (half == 0) {
#pragma unroll
          for (int i = 0; i < RSLOTS; ++i) qk_sm(i, dK + i * U_CH, i == 0 ? 0u : 1u);
        } else {
#pragma unroll
          for (int i = 0; i < NVC; ++i) qk_tm(i, dK + i * U_CH, i == 0 ? 0u : 1u);
          qk_sm(NQS - 1, dK + NVC * U_CH, 1u);
        }
        mma_commit(&B->r_empty);               // the ring may be refilled
        if (!(ok = wait_bar(B, &B->v_full, ph, P.status))) break;
        tc_fence_after();
        if (half == 0) {
#pragma unroll
          for (int i = 0; i < NVC; ++i) qk_tm(i, dVk + i * U_CH, 1u);
        } else {
#pragma unroll
          for (int i = 0; i < NVC; ++i) qk_sm(i, dVk + i * U_CH, 1u);
        }
        mma_commit(&B->s_full);
        // O += P(t) V(t)
        if (!(ok = wait_bar(B, &B->p_full, ph, P.status))) break;
        tc_fence_after();
        const uint32_t acc0 = t ? 1u : 0u;
        mma_f16_ts(tO, tP, dv, idesc_pv, acc0);
#pragma unroll
        for (int k = 1; k < KT / 16; ++k)   // 16 keys per MMA: 8 P columns, 16 V rows
          mma_f16_ts(tO, tP + 8 * k, dv + (uint64_t)U_KSTEP * k, idesc_pv, 1u);
        mma_commit(&B->o_done);
      }
      // no MMA of this CTA may still run when its tensor memory is freed
      mma_commit(&B->drain);
      mbar_wait(&B->drain, 0, P.status);
    }
  } else {
    softmax_and_stage(P, B, smem, tmem, b, qt, row0, kvl, W, j_lo, nt);
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (P.splits > 1) cluster_sync_all();   // every split's partial is staged
  tc_fence_after();
  if (warp == 5) tmem_dealloc(tmem, TMEM_COLS);
  reduce_splits(P, smem, half, split, b, qt, row0);
  cluster_sync_all();          // no CTA leaves while another may still read its staged partial
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
                              float* lse, bool pdl) {
  const Layout& l = h->lay;
  const int ps = h->cfg.page_size;
  if (l.rkv != 512 || l.dr != 64)
    return fail(MLA_ERR_UNSUPPORTED, "tcgen05 attention: needs kv_lora_rank 512, qk_rope_head_dim 64");
  if (ps % 16 || (ps < KT && KT % ps) || (ps > KT && ps % KT))
    return fail(MLA_ERR_UNSUPPORTED, "tcgen05 attention: page_size must be 16, 32, 64 or a multiple of 128");
  if (d.num_blocks <= 0) return MLA_OK;
  const int splits = attn_splits(h, d.num_blocks, d.block_len);
  AttnParams P;
  const long rows = (long)d.num_blocks * d.block_len * l.H;
  const long slots = (long)num_pages * ps;
  if (!make_tmap_chunked(&P.tmQ, false, q_abs, rows, l.L, l.L, QROWS, NQS) ||
      !make_tmap_2d(&P.tmK, false, cache, slots, l.L, l.L, KT) ||
      !make_tmap_2d(&P.tmKs, false, cache, slots, l.L, l.L, ps < KT ? ps : KT) ||
      !make_tmap_chunked(&P.tmV, false, cache, slots, l.L, l.L, KT, 4))
    return fail(MLA_ERR_CUDA, "tcgen05 attention: cuTensorMapEncodeTiled failed");
  P.q_abs = q_abs;
  P.block_table = d.block_table;
  P.kv_len = d.kv_len;
  P.window = d.window;
  P.q_visible = d.q_visible;
  P.positions = positions;
  P.vis_stats = d.vis_stats;
  P.o_lat = o_lat;
  P.lse = lse;
  P.status = h->status;
  P.max_pages = d.max_pages;
  P.num_pages = num_pages;
  P.page_size = ps;
  P.seg_rows = ps < KT ? ps : KT;
  P.T = d.block_len;
  P.H = l.H;
  P.tiles_per_block = (d.block_len * l.H + QROWS - 1) / QROWS;
  P.scale_log2 = h->scale * 1.4426950408889634f;
  P.splits = splits;
  static std::once_flag once;
  std::call_once(once, [] {
    cudaFuncSetAttribute(latent_attn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
  });
  Launch L(dim3(2 * d.num_blocks * P.tiles_per_block, splits, 1), dim3(THREADS), SMEM_BYTES, st, pdl,
           dim3(2, splits, 1));
  const cudaError_t e = cudaLaunchKernelEx(&L.cfg, latent_attn_tc_kernel, P);
  if (e != cudaSuccess) return cuda_fail(e, "tcgen05 attention launch");
  return MLA_OK;
}

// When the (block, 128-row, value-half) CTAs leave part of the GPU idle
// (one CTA per SM), split each unit's key range so that the CTAs fill one
// wave (at most MAX_SPLITS parts: a unit's CTAs form one cluster); a split
// that would add a partial wave only lengthens the kernel.
int attn_splits(const mla_handle* h, long num_blocks, int block_len) {
  const long ctas = 2 * num_blocks * ((block_len * h->lay.H + QROWS - 1) / QROWS);
  const long wave = h->num_sms;
  if (ctas <= 0 || ctas >= wave) return 1;
  const long s = wave / ctas;
  return (int)(s < 1 ? 1 : s > MAX_SPLITS ? MAX_SPLITS : s);
}

}  // namespace tc
}  // namespace mla
