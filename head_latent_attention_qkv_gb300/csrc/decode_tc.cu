// tcgen05 latent attention for blocks of few query rows (the cached decode
// of one token per sequence: "MLA (Multi-Head Latent Attention)" blog,
// forward_mqa / decode_attention_fwd, whose key range is split across the
// SMs (num_kv_splits) and merged by log-sum-exp).
//
// With at most 32 query rows per block, a 128-row query tile would be three
// quarters padding.  Here the roles are transposed: 128 keys of the cache
// fill the MMA's M dimension and the block's rows its N dimension (N = 32),
//   S^T = K Q^T        (M = 128 keys, N = 32 rows, K = 576 dims; 36 MMAs)
//   O^T += V^T P^T     (M = 128 value dims x 4, N = 32 rows, K = 128 keys; 32 MMAs)
// so one CTA holds all 512 value dims of its rows in 4 x 32 tensor-memory
// columns and computes every score once.  The A operand of the second
// product is the cache chunk itself read MN-major (value dims contiguous);
// P^T is the B operand, written by the softmax into shared memory as P
// [row][key] (K-major, 128-byte swizzle).
//
// Work unit: (block, key split).  A split covers `tiles_per_split` 128-key
// tiles; every split writes its normalised partial output (fp32), its
// log2-sum-exp and visibility counts into the workspace, and the merge
// kernel combines the splits of a block in split order (the blog's
// forward_mha merge_attn_states).  Splits are many and short (about four
// tiles) so that the SMs stay busy whatever the mix of sequence lengths.
//
// Shared memory: the nine 64-dim chunks of one key tile (one slot each,
// slot c = chunk c), Q (nine chunks of 32 rows), P (two 64-key chunks).
// Per tile the tensor pipe runs S^T over chunks 8, 0-3 (group A), 4-5 (B),
// 6-7 (C), then, once the softmax has written P, O^T by value group 0..3;
// each group's chunks are refilled for the next tile as soon as the O^T
// group that reads them is done (chunk 8 with group A), so the next tile's
// copies run under the current tile's O^T.
//   warps 0-3 : softmax, thread = key (TMEM lane); row maxima by a butterfly
//               transpose reduction across the warp and a 4-warp combine;
//               running max per row kept identically by every thread (lazy
//               rescale beyond 2^8); row sums kept per thread until the end
//   warp 4    : page rows, Q, group A copies      warp 6: groups B, C copies
//   warp 5    : tensor-memory allocation, MMA issue
#include "decode_tc.cuh"

#include <mutex>

#include "gemm_tc.cuh"
#include "tc_ptx.cuh"

namespace mla {
namespace tc {
namespace {

constexpr int KT = 128, DCH = 64, NCH = 9, NR = 32;   // keys per tile, dims per chunk, rows (N)
constexpr int THREADS = 224;                           // softmax x4, TMA, MMA, TMA
constexpr int KV_CH_BYTES = KT * DCH * 2;              // 16 KiB
constexpr int Q_CH_BYTES = NR * DCH * 2;               // 4 KiB
constexpr int P_CH_BYTES = NR * DCH * 2;               // 4 KiB (64 keys)
constexpr int OFF_K = 0;
constexpr int OFF_Q = OFF_K + NCH * KV_CH_BYTES;
constexpr int OFF_P = OFF_Q + NCH * Q_CH_BYTES;
constexpr int OFF_RED = OFF_P + 2 * P_CH_BYTES;        // reduction scratch
constexpr int OFF_BAR = OFF_RED + 2048;
constexpr int SMEM_BYTES = 1024 + OFF_BAR + 256;
constexpr uint32_t TMEM_COLS = 256, TM_S = 0, TM_O = 32;    // O^T group g at TM_O + 32 g
constexpr float RESCALE_LOG2 = 8.f;
static_assert(SMEM_BYTES <= 232448, "shared memory");

struct Bars {
  uint64_t q_full;
  uint64_t g_full[3];      // key chunks landed: A = {8, 0..3}, B = {4, 5}, C = {6, 7} (phase t)
  uint64_t g_empty[3];     // the MMAs reading the group are done (phase t)
  uint64_t s_full;         // S^T(t) complete (and O^T(t - 1): same issuing thread)
  uint64_t p_full;         // P(t) in shared memory (128 arrivals)
  uint64_t o_done;         // O^T(t) complete
  uint64_t drain;
  uint32_t tmem_slot;
  int abort;
};
static_assert(sizeof(Bars) <= 256, "barrier block");

__device__ __forceinline__ bool wait_bar(Bars* B, uint64_t* bar, uint32_t parity, uint32_t* st) {
  if (*(volatile int*)&B->abort) return false;
  if (mbar_wait(bar, parity, st)) return true;
  B->abort = 1;
  return false;
}
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ void softmax_sync() { asm volatile("bar.sync 2, 128;" ::: "memory"); }

// Lane l of the warp ends with op over the warp's 32 lanes of x[l] (x[0..31]
// per lane); 31 shuffles.
template <bool kMax>
__device__ __forceinline__ float warp_transpose_reduce(float* x, int lane) {
#pragma unroll
  for (int s = 16; s >= 1; s >>= 1) {
    const bool upper = (lane & s) != 0;
#pragma unroll
    for (int i = 0; i < s; ++i) {
      const float lo = x[i], hi = x[i + s];
      const float send = upper ? lo : hi, keep = upper ? hi : lo;
      const float recv = __shfl_xor_sync(0xffffffffu, send, s);
      x[i] = kMax ? fmaxf(keep, recv) : keep + recv;
    }
  }
  return x[0];
}

__global__ void __launch_bounds__(THREADS, 1) latent_decode_tc_kernel(const __grid_constant__ DecodeParams P) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  Bars* B = (Bars*)(smem + OFF_BAR);
  float* red = (float*)(smem + OFF_RED);     // [2][4][32] warp partials, [32] combined, [32] rows' lo/hi
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  const int b = blockIdx.x / P.splits, split = blockIdx.x % P.splits;
  const int R = P.T * P.H;                                  // live rows (<= 32)
  const long row0 = (long)b * R;                           // first Q_abs row of the block

  int kvl = P.kv_len[b];
  const int cap = P.max_pages * P.page_size;
  if (kvl < 0 || kvl > cap) {
    if (tid == 0 && split == 0) set_status(P.status, MLA_DEV_BAD_LENGTH);
    kvl = max(0, min(kvl, cap));
  }
  const int W = P.window ? P.window[b] : 0;
  if (W < 0) {
    if (tid == 0 && split == 0) set_status(P.status, MLA_DEV_BAD_WINDOW);
    kvl = 0;
  }
  // key range of the block: [j_lo, kvl) from the first key any row sees
  int j_lo = 0;
  if (W > 0) {
    int pmin = 0x7fffffff;
    for (int t = 0; t < P.T; ++t) pmin = min(pmin, P.positions[(long)b * P.T + t]);
    j_lo = max(0, pmin - W + 1) / KT * KT;
  }
  const int nt_all = kvl > j_lo ? (kvl - j_lo + KT - 1) / KT : 0;
  const int t_begin = split * P.tiles_per_split;
  const int nt = max(0, min(nt_all, t_begin + P.tiles_per_split) - t_begin);
  const int k_begin = j_lo + t_begin * KT;                // first key of this split
  const int k_end = min(kvl, k_begin + nt * KT);
  const long part_base = ((long)b * P.splits + split) * NR;   // partial rows of this split
  if (nt == 0) {
    // a split past the block's keys: an empty partial the merge skips
    pdl_wait();
    if (tid < R) P.part_lse[part_base + tid] = -INFINITY;
    if (tid < P.T) {
      int* vs = P.part_vis + (((long)b * P.splits + split) * P.T + tid) * 3;
      vs[0] = 0; vs[1] = -1; vs[2] = -1;
    }
    return;
  }

  if (tid == 0) {
    mbar_init(&B->q_full, 1);
    for (int g = 0; g < 3; ++g) {
      mbar_init(&B->g_full[g], 1);
      mbar_init(&B->g_empty[g], 1);
    }
    mbar_init(&B->s_full, 1);
    mbar_init(&B->p_full, 128);
    mbar_init(&B->o_done, 1);
    mbar_init(&B->drain, 1);
    B->abort = 0;
    fence_mbar_init();
  }
  if (warp == 5) tmem_alloc(&B->tmem_slot, TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = B->tmem_slot;
  if (tid == 0) pdl_trigger();
  pdl_wait();

  if (warp == 4 || warp == 6) {
    if (lane == 0 && nt > 0) {
      const int ps = P.page_size, past_end = P.num_pages * ps;
      // first cache row of tile t (past_end for an invalid page: zeros)
      auto tile_row = [&](int t) {
        const int j0 = k_begin + t * KT;
        const int pg = P.block_table[(long)b * P.max_pages + j0 / ps];
        if (pg < 0 || pg >= P.num_pages) {
          set_status(P.status, MLA_DEV_BAD_PAGE);
          return past_end;
        }
        return pg * ps + j0 % ps;
      };
      bool ok = true;
      if (warp == 4) {
        prefetch_tmap(&P.tmQ);
        prefetch_tmap(&P.tmK1);
        prefetch_tmap(&P.tmK4);
        mbar_arrive_expect_tx(&B->q_full, NCH * Q_CH_BYTES);
        tma_load_3d(smem + OFF_Q, &P.tmQ, &B->q_full, 0, (int)row0, 0);
        for (int t = 0; t < nt && ok; ++t) {
          if (!(ok = wait_bar(B, &B->g_empty[0], (t & 1) ^ 1, P.status))) break;
          const int y0 = tile_row(t);
          mbar_arrive_expect_tx(&B->g_full[0], 5 * KV_CH_BYTES);
          tma_load_3d(smem + OFF_K + 8 * KV_CH_BYTES, &P.tmK1, &B->g_full[0], 8 * DCH, y0, 0);
          tma_load_3d(smem + OFF_K, &P.tmK4, &B->g_full[0], 0, y0, 0);
        }
        mbar_wait(&B->q_full, 0, P.status);
        mbar_wait(&B->g_full[0], (nt - 1) & 1, P.status);
      } else {
        prefetch_tmap(&P.tmK2);
        for (int t = 0; t < nt && ok; ++t) {
          const int y0 = tile_row(t);
          for (int g = 1; g < 3 && ok; ++g) {
            if (!(ok = wait_bar(B, &B->g_empty[g], (t & 1) ^ 1, P.status))) break;
            mbar_arrive_expect_tx(&B->g_full[g], 2 * KV_CH_BYTES);
            tma_load_3d(smem + OFF_K + (2 + 2 * g) * KV_CH_BYTES, &P.tmK2, &B->g_full[g], 0, y0, 2 + 2 * g);
          }
        }
        for (int g = 1; g < 3; ++g) mbar_wait(&B->g_full[g], (nt - 1) & 1, P.status);
      }
    }
  } else if (warp == 5) {
    if (lane == 0 && nt > 0) {
      // ---- MMA issuer ----
      const uint32_t idesc_s = idesc_f16(128, NR, false);                 // K-major A and B
      const uint32_t idesc_o = idesc_f16(128, NR, false) | (1u << 15);    // A (V^T) MN-major
      bool ok = wait_bar(B, &B->q_full, 0, P.status);
      auto s_chunk = [&](int c, bool first) {
        const uint64_t da = smem_desc_sw128(smem + OFF_K + c * KV_CH_BYTES);
        const uint64_t db = smem_desc_sw128(smem + OFF_Q + c * Q_CH_BYTES);
#pragma unroll
        for (int k = 0; k < DCH / 16; ++k)
          mma_f16(tmem + TM_S, da + 2 * k, db + 2 * k, idesc_s, !(first && k == 0));
      };
      auto o_group = [&](int g, bool first_tile) {
        const uint64_t da = smem_desc_sw128_mn(smem + OFF_K + 2 * g * KV_CH_BYTES, KV_CH_BYTES);
#pragma unroll
        for (int k = 0; k < KT / 16; ++k) {
          const uint64_t db = smem_desc_sw128(smem + OFF_P + (k / 4) * P_CH_BYTES) + 2 * (k % 4);
          mma_f16(tmem + TM_O + 32 * g, da + (uint64_t)(16 * 128 / 16) * k, db, idesc_o,
                  !(first_tile && k == 0));
        }
      };
      for (int t = 0; t < nt && ok; ++t) {
        const uint32_t ph = t & 1;
        if (!(ok = wait_bar(B, &B->g_full[0], ph, P.status))) break;
        tc_fence_after();
        s_chunk(8, true);
#pragma unroll 1
        for (int c = 0; c < 4; ++c) s_chunk(c, false);
        if (!(ok = wait_bar(B, &B->g_full[1], ph, P.status))) break;
        tc_fence_after();
        s_chunk(4, false);
        s_chunk(5, false);
        if (!(ok = wait_bar(B, &B->g_full[2], ph, P.status))) break;
        tc_fence_after();
        s_chunk(6, false);
        s_chunk(7, false);
        mma_commit(&B->s_full);
        if (!(ok = wait_bar(B, &B->p_full, ph, P.status))) break;
        tc_fence_after();
        o_group(0, t == 0);
        o_group(1, t == 0);
        mma_commit(&B->g_empty[0]);
        o_group(2, t == 0);
        mma_commit(&B->g_empty[1]);
        o_group(3, t == 0);
        mma_commit(&B->g_empty[2]);
        mma_commit(&B->o_done);
      }
      mma_commit(&B->drain);
      mbar_wait(&B->drain, 0, P.status);
    }
  } else {
    // ---- softmax warps: thread k = key k of the tile (TMEM lane k) ----
    const int k = tid;
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    float* wpart = red;                     // [2][4][32]
    float* comb = red + 256;                // [32] combined row values
    int* rlo = (int*)(red + 288);           // [32] first visible key of each row
    int* rhi = (int*)(red + 320);           // [32] end of each row's visible keys
    if (k < NR) {
      int lo = 0, hi = 0;
      if (k < R) {
        const long m = (long)b * P.T + k / P.H;
        const int p = P.positions[m];
        const bool qv = P.q_visible ? P.q_visible[m] != 0 : true;
        lo = W > 0 ? max(0, p - W + 1) : 0;
        hi = qv ? kvl : 0;
      }
      rlo[k] = lo;
      rhi[k] = hi;
    }
    softmax_sync();
    float mrow[NR], lrow[NR];
#pragma unroll
    for (int r = 0; r < NR; ++r) { mrow[r] = -INFINITY; lrow[r] = 0.f; }
    for (int t = 0; t < nt; ++t) {
      const uint32_t ph = t & 1;
      const int j = k_begin + t * KT + k;   // this thread's key
      float s[NR];
      wait_bar(B, &B->s_full, ph, P.status);
      tc_fence_after();
      tmem_ld32_nowait(tmem + TM_S + lane_base, s);
      tmem_ld_wait();
      tmem_reg_fence32(s);
      // mask by logical position: row r sees keys [rlo, rhi)
#pragma unroll
      for (int r = 0; r < NR; ++r) s[r] = (j >= rlo[r] && j < rhi[r]) ? s[r] : -INFINITY;
      float x[NR];
#pragma unroll
      for (int r = 0; r < NR; ++r) x[r] = s[r];
      const float wmax = warp_transpose_reduce<true>(x, lane);   // lane l: max of row l over the warp
      wpart[ph * 128 + warp * 32 + lane] = wmax;
      softmax_sync();
      if (warp == 0) {
        const float* w4 = wpart + ph * 128;
        comb[lane] = fmaxf(fmaxf(w4[lane], w4[32 + lane]), fmaxf(w4[64 + lane], w4[96 + lane]));
      }
      softmax_sync();
      // every thread updates the rows' running maxima identically (exp2 domain)
      float alpha[NR];
      bool any_rescale = false;
#pragma unroll
      for (int r = 0; r < NR; ++r) {
        const float tm = comb[r] * P.scale_log2;
        const bool grow = tm > mrow[r] + RESCALE_LOG2;
        const float m_new = grow ? tm : mrow[r];
        alpha[r] = (grow && mrow[r] != -INFINITY) ? exp2f(mrow[r] - m_new) : 1.f;
        any_rescale |= alpha[r] != 1.f;
        mrow[r] = m_new;
      }
      // value rows of keys past kv_len may hold anything: zero this key's
      // row in the eight value chunks before P V^T reads them
      if (j >= kvl) {
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          uint4* rowp = reinterpret_cast<uint4*>(smem + OFF_K + c * KV_CH_BYTES + k * 128);
#pragma unroll
          for (int q = 0; q < 8; ++q) rowp[q] = make_uint4(0, 0, 0, 0);
        }
      }
      // P[r][k] (bf16) into the swizzled K-major tile: 16-byte unit (k % 64) / 8
      // of row r sits at unit ((k % 64) / 8) ^ (r % 8)
      uint8_t* pchunk = smem + OFF_P + (k / 64) * P_CH_BYTES;
      const int kk = k % 64;
#pragma unroll
      for (int r = 0; r < NR; ++r) {
        const float mref = mrow[r] == -INFINITY ? 0.f : mrow[r];
        const float p = fast_exp2(fmaf(s[r], P.scale_log2, -mref));
        lrow[r] = lrow[r] * alpha[r] + p;
        *reinterpret_cast<__nv_bfloat16*>(pchunk + r * 128 + (((kk >> 3) ^ (r & 7)) << 4) + (kk & 7) * 2) =
            __float2bfloat16_rn(p);
      }
      // O^T(t - 1) has completed (before S^T(t)): rescale the rows that grew
      if (t > 0 && __any_sync(0xffffffffu, any_rescale)) {
#pragma unroll 1
        for (int g = 0; g < 4; ++g) {
          float o[NR];
          tmem_ld32_nowait(tmem + TM_O + 32 * g + lane_base, o);
          tmem_ld_wait();
          tmem_reg_fence32(o);
#pragma unroll
          for (int r = 0; r < NR; ++r) o[r] *= alpha[r];
          tmem_st32(tmem + TM_O + 32 * g + lane_base, o);
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&B->p_full);
    }
    // rows' sums over the 128 keys of every tile (threads hold partials)
    float x[NR];
#pragma unroll
    for (int r = 0; r < NR; ++r) x[r] = lrow[r];
    const float wsum = warp_transpose_reduce<false>(x, lane);
    softmax_sync();
    wpart[warp * 32 + lane] = wsum;
    softmax_sync();
    if (warp == 0) comb[lane] = (wpart[lane] + wpart[32 + lane]) + (wpart[64 + lane] + wpart[96 + lane]);
    softmax_sync();
    if (nt > 0) wait_bar(B, &B->o_done, (nt - 1) & 1, P.status);
    tc_fence_after();
    // partial output of this split: thread k holds value dim 128 g + k of every row
#pragma unroll 1
    for (int g = 0; g < 4; ++g) {
      float o[NR];
      if (nt > 0) {
        tmem_ld32_nowait(tmem + TM_O + 32 * g + lane_base, o);
        tmem_ld_wait();
        tmem_reg_fence32(o);
      }
#pragma unroll
      for (int r = 0; r < NR; ++r) {
        const float l = comb[r];
        if (r < R) P.part[(part_base + r) * 512 + 128 * g + k] = (nt > 0 && l > 0.f) ? o[r] / l : 0.f;
      }
    }
    float mk = -INFINITY;                   // row k's running max (registers indexed statically)
#pragma unroll
    for (int r = 0; r < NR; ++r) mk = (r == k) ? mrow[r] : mk;
    if (k < R) P.part_lse[part_base + k] = (nt > 0 && comb[k] > 0.f) ? mk + log2f(comb[k]) : -INFINITY;
    if (k < P.T) {   // visibility of token k over this split's keys (one interval)
      const int lo = max(rlo[k * P.H], k_begin), hi = min(rhi[k * P.H], k_end);
      int* vs = P.part_vis + (((long)b * P.splits + split) * P.T + k) * 3;
      vs[0] = hi > lo ? hi - lo : 0;
      vs[1] = hi > lo ? lo : -1;
      vs[2] = hi > lo ? hi - 1 : -1;
    }
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 5) tmem_dealloc(tmem, TMEM_COLS);
}

// One CTA per (block, row): the splits' partials of the row combined by
// log-sum-exp in split order (empty splits, lse = -inf, skipped); a row no
// split saw stays exactly zero.  Thread i handles value dims 4i .. 4i + 3.
constexpr int MERGE_THREADS = 128, MAX_MERGE_SPLITS = 64;
__global__ void __launch_bounds__(MERGE_THREADS) decode_merge_kernel(const __grid_constant__ DecodeParams P) {
  const int R = P.T * P.H;
  const int b = blockIdx.x / R, r = blockIdx.x % R;
  const long base = (long)b * P.splits * NR + r;          // partial row of split s: base + s * NR
  __shared__ float w_s[MAX_MERGE_SPLITS];
  __shared__ float den_s, mx_s;
  if (threadIdx.x < 32) {
    float mx = -INFINITY;
    for (int s = threadIdx.x; s < P.splits; s += 32) mx = fmaxf(mx, P.part_lse[base + s * NR]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    float den = 0.f;
    for (int s = threadIdx.x; s < P.splits; s += 32) {
      const float l = P.part_lse[base + s * NR];
      const float w = (mx == -INFINITY || l == -INFINITY) ? 0.f : exp2f(l - mx);
      w_s[s] = w;
      den += w;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
    if (threadIdx.x == 0) { den_s = den; mx_s = mx; }
  }
  __syncthreads();
  const float den = den_s;
  const int d = 4 * threadIdx.x;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int s = 0; s < P.splits; ++s) {
    const float w = w_s[s];
    if (w == 0.f) continue;
    const float4 v = *reinterpret_cast<const float4*>(P.part + (base + s * NR) * 512 + d);
    acc.x += w * v.x; acc.y += w * v.y; acc.z += w * v.z; acc.w += w * v.w;
  }
  const float inv = den > 0.f ? 1.f / den : 0.f;
  const long row = (long)b * R + r;
  __half2 h2[2] = {__floats2half2_rn(acc.x * inv, acc.y * inv), __floats2half2_rn(acc.z * inv, acc.w * inv)};
  *reinterpret_cast<uint2*>(P.o_lat + row * 512 + d) = *reinterpret_cast<uint2*>(h2);
  if (threadIdx.x == 0 && P.lse) P.lse[row] = den > 0.f ? (mx_s + log2f(den)) * 0.6931471805599453f : -INFINITY;
  // visibility statistics of the row's token (from its head-0 row)
  if (threadIdx.x == 0 && P.vis_stats && r % P.H == 0) {
    const int t = r / P.H;
    int cnt = 0, first = -1, last = -1;
    for (int s = 0; s < P.splits; ++s) {
      const int* vs = P.part_vis + (((long)b * P.splits + s) * P.T + t) * 3;
      if (vs[0] > 0) {
        first = cnt ? min(first, vs[1]) : vs[1];
        last = max(last, vs[2]);
        cnt += vs[0];
      }
    }
    const long m = (long)b * P.T + t;
    P.vis_stats[m * 3 + 0] = cnt;
    P.vis_stats[m * 3 + 1] = cnt ? first : -1;
    P.vis_stats[m * 3 + 2] = cnt ? last : -1;
  }
}

}  // namespace

bool decode_applies(const mla_handle* h, int block_len) {
  const Layout& l = h->lay;
  return h->cfg.dtype == MLA_BF16 && l.rkv == 512 && l.dr == 64 && block_len * l.H <= NR &&
         h->cfg.page_size % KT == 0;
}

static int tiles_per_split(const mla_handle* h, const mla_attn_desc_t& d) {
  const int max_tiles = (d.max_pages * h->cfg.page_size + KT - 1) / KT;
  // about four CTAs per SM over the launch, each on a short key range
  const long units = (long)d.num_blocks * max_tiles;
  const long target = 4L * h->num_sms;
  long tps = (units + target - 1) / target;
  if (tps < 1) tps = 1;
  if (tps > max_tiles) tps = max_tiles;
  // the merge holds at most MAX_MERGE_SPLITS splits of a block
  const long min_tps = (max_tiles + MAX_MERGE_SPLITS - 1) / MAX_MERGE_SPLITS;
  if (tps < min_tps) tps = min_tps;
  return (int)tps;
}

size_t decode_workspace_bytes(const mla_handle* h, const mla_attn_desc_t& d) {
  const int max_tiles = (d.max_pages * h->cfg.page_size + KT - 1) / KT;
  const int tps = tiles_per_split(h, d);
  const long splits = (max_tiles + tps - 1) / tps;
  const long parts = (long)d.num_blocks * splits;
  return align256(parts * NR * 512 * 4) + align256(parts * NR * 4) +
         align256(parts * d.block_len * 3 * 4);
}

mla_status_t latent_decode(cudaStream_t st, const mla_handle* h, const __nv_bfloat16* q_abs,
                           const __nv_bfloat16* cache, int num_pages, const mla_attn_desc_t& d,
                           const int32_t* positions, __half* o_lat, float* lse, void* workspace,
                           size_t workspace_bytes, bool pdl) {
  const Layout& l = h->lay;
  if (!decode_applies(h, d.block_len))
    return fail(MLA_ERR_UNSUPPORTED, "decode attention: needs block_len * num_heads <= 32, page_size a multiple of 128");
  if (d.num_blocks <= 0) return MLA_OK;
  if (workspace_bytes < decode_workspace_bytes(h, d) || (uintptr_t)workspace % 256)
    return fail(MLA_ERR_INVALID_ARG, "decode attention: workspace too small or not 256-byte aligned");
  DecodeParams P;
  const long rows = (long)d.num_blocks * d.block_len * l.H;
  const long slots = (long)num_pages * h->cfg.page_size;
  if (!make_tmap_chunked(&P.tmQ, false, q_abs, rows, l.L, l.L, NR, NCH) ||
      !make_tmap_2d(&P.tmK1, false, cache, slots, l.L, l.L, KT) ||
      !make_tmap_chunked(&P.tmK2, false, cache, slots, l.L, l.L, KT, 2) ||
      !make_tmap_chunked(&P.tmK4, false, cache, slots, l.L, l.L, KT, 4))
    return fail(MLA_ERR_CUDA, "decode attention: cuTensorMapEncodeTiled failed");
  const int max_tiles = (d.max_pages * h->cfg.page_size + KT - 1) / KT;
  P.tiles_per_split = tiles_per_split(h, d);
  P.splits = (max_tiles + P.tiles_per_split - 1) / P.tiles_per_split;
  const long parts = (long)d.num_blocks * P.splits;
  char* ws = (char*)workspace;
  P.part = (float*)ws;
  P.part_lse = (float*)(ws + align256(parts * NR * 512 * 4));
  P.part_vis = (int*)(ws + align256(parts * NR * 512 * 4) + align256(parts * NR * 4));
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
  P.page_size = h->cfg.page_size;
  P.T = d.block_len;
  P.H = l.H;
  P.scale_log2 = h->scale * 1.4426950408889634f;
  static std::once_flag once;
  std::call_once(once, [] {
    cudaFuncSetAttribute(latent_decode_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
  });
  Launch L(dim3((unsigned)parts), dim3(THREADS), SMEM_BYTES, st, pdl);
  cudaError_t e = cudaLaunchKernelEx(&L.cfg, latent_decode_tc_kernel, P);
  if (e != cudaSuccess) return cuda_fail(e, "decode attention launch");
  decode_merge_kernel<<<d.num_blocks * d.block_len * l.H, MERGE_THREADS, 0, st>>>(P);
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "decode merge launch");
  return MLA_OK;
}

}  // namespace tc
}  // namespace mla
