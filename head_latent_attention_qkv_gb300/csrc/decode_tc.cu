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
// Work split: one persistent CTA per SM.  The U 128-key tiles of all blocks,
// in block order, are cut into G = min(gridDim.x, U) equal ranges (none
// empty); CTA c < G takes range c, which covers the tail of one block, whole
// blocks and the head of another.  Each (block, CTA) piece is a segment; it
// writes its normalised partial output (fp32), log2-sum-exp and visibility
// counts to partial slot block + c (distinct for every segment: along the
// tile order neither the block nor the CTA ever decreases and one of them
// grows), and the merge kernel combines the segments of a block in CTA order
// (the blog's forward_mha merge_attn_states).
//
// Pipeline.  The tensor pipe runs, per segment of n tiles,
//   S^T(0) S^T(1) O^T(0) S^T(2) O^T(1) ... S^T(n-1) O^T(n-2) O^T(n-1)
// so the scores of tile t + 1 are computed while the softmax of tile t runs
// (S^T and P double-buffered).  The cache streams through a ring of five
// 32 KiB slots (two 64-dim chunks each) in exactly that order: per tile the
// key items (chunk pairs 0-1, 2-3, 4-5, 6-7, then the rope chunk 8) and, one
// tile later, the value items (pairs 0-1 .. 6-7, read again, now from L2).
//   warps 0-3 : softmax, thread = key (TMEM lane); row maxima by a butterfly
//               transpose reduction across the warp and a 4-warp combine;
//               each row's running max and rescale factor kept once in
//               shared memory (lazy rescale beyond 2^8); segment epilogue
//   warp 4    : tensor-memory allocation, MMA issue
//   warps 5-6 : ring copies (slots 0, 2, 4 / slots 1, 3)
//   warp 7    : Q of each segment; zeroes the value rows past kv_len of a
//               block's last tile (they may hold anything) before O^T reads them
#include "decode_tc.cuh"

#include <mutex>

#include "gemm_tc.cuh"
#include "tc_ptx.cuh"

namespace mla {
namespace tc {
namespace {

constexpr int KT = 128, DCH = 64, NCH = 9, NR = 32;   // keys per tile, dims per chunk, rows (N)
constexpr int THREADS = 256;
constexpr int NSLOT = 5;                               // ring slots (chunk pairs)
constexpr int KV_CH_BYTES = KT * DCH * 2;              // 16 KiB
constexpr int SLOT_BYTES = 2 * KV_CH_BYTES;            // 32 KiB
constexpr int Q_CH_BYTES = NR * DCH * 2;               // 4 KiB
constexpr int P_CH_BYTES = NR * DCH * 2;               // 4 KiB (64 keys)
constexpr int P_BYTES = 2 * P_CH_BYTES;                // one tile's P
constexpr int K_ITEMS = 5, V_ITEMS = 4;                // ring items per tile
constexpr int OFF_RING = 0;
constexpr int OFF_Q = OFF_RING + NSLOT * SLOT_BYTES;
constexpr int OFF_P = OFF_Q + NCH * Q_CH_BYTES;
constexpr int OFF_RED = OFF_P + 2 * P_BYTES;
constexpr int RED_BYTES = 2048;
constexpr int OFF_BAR = OFF_RED + RED_BYTES;
constexpr int SMEM_BYTES = 1024 + OFF_BAR + 256;
// TMEM: S^T double buffer by tile (2 x 32 columns), O^T double buffer by segment (2 x 128)
constexpr uint32_t TMEM_COLS = 512, TM_S = 0, TM_O = 64;
constexpr float RESCALE_LOG2 = 8.f;
static_assert(SMEM_BYTES <= 232448, "shared memory");

// shared reduction area (4-byte words)
constexpr int RD_WPART = 0;      // [4][32] per-warp row values
constexpr int RD_M = 128;        // [32] running row max (log2 domain)
constexpr int RD_ALPHA = 160;    // [32] rescale factor of the current tile
constexpr int RD_INVL = 192;     // [32] 1 / row sum
constexpr int RD_LO = 224;       // [32] first visible key of each row
constexpr int RD_HI = 256;       // [32] end of each row's visible keys
constexpr int RD_FLAG = 288;     // some row rescaled in this tile
constexpr int RD_SCH = 320;      // [8] scan partials, [12..13] first block / tile of the range
static_assert((RD_SCH + 16) * 4 <= RED_BYTES, "reduction area");

// Every barrier is waited on phase by phase by its one consumer role, and
// the producer side can run at most one phase ahead of that wait (the
// parity test tells only two consecutive phases apart).  Hence the S^T and
// P barriers are doubled by tile parity (S^T(g + 1) may complete before the
// softmax of tile g starts), the epilogue has its own per-segment barrier,
// and the value rows past kv_len are zeroed only after the MMA thread, which
// waits on every phase of the ring in order, hands their items over.
struct Bars {
  uint64_t full[NSLOT];    // ring slot landed
  uint64_t empty[NSLOT];   // the MMAs reading the slot are done
  uint64_t vready;         // a block's last (ragged) tile: its value items landed
  uint64_t vfix;           // ... and their rows past kv_len are zeroed
  uint64_t q_full, q_empty;
  uint64_t s_full[2];      // S^T(g) complete (and every MMA issued before it), by g % 2
  uint64_t p_full[2];      // P(g) in shared memory (128 arrivals), by g % 2
  uint64_t o_done;         // O^T(g) complete (waited on only for a rescale)
  uint64_t o_seg;          // the segment's last O^T complete
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

// Key range of block b: [j_lo, kvl), j_lo the first key any of its rows can
// see under the sliding window, rounded down to a tile; nt tiles.  kv_len
// outside [0, max_pages * page_size] is clamped and a negative window empties
// the block (both reported once, by the first CTA).
struct BlockKeys {
  int kvl, j_lo, W, nt;
  bool bad_len, bad_win;
};
__device__ __forceinline__ BlockKeys block_keys(const DecodeParams& P, int b) {
  BlockKeys k;
  int kvl = P.kv_len[b];
  const int cap = P.max_pages * P.page_size;
  k.bad_len = kvl < 0 || kvl > cap;
  kvl = max(0, min(kvl, cap));
  k.W = P.window ? P.window[b] : 0;
  k.bad_win = k.W < 0;
  if (k.bad_win) kvl = 0;
  k.j_lo = 0;
  if (k.W > 0) {
    int pmin = 0x7fffffff;
    for (int t = 0; t < P.T; ++t) pmin = min(pmin, P.positions[(long)b * P.T + t]);
    k.j_lo = max(0, pmin - k.W + 1) / KT * KT;
  }
  k.kvl = kvl;
  k.nt = kvl > k.j_lo ? (kvl - k.j_lo + KT - 1) / KT : 0;
  return k;
}

// The CTA whose tile range [c U / G, (c + 1) U / G) holds global tile u
// (G <= U: no range is empty).
__device__ __forceinline__ int cta_of(long long u, long long U, int G) {
  return (int)(((u + 1) * G - 1) / U);
}

// Segments of this CTA's range, in order: tiles [t0, t0 + n) of block b.
struct Seg {
  int b, t0, n;
  BlockKeys k;
};
struct SegIter {
  int b, t;        // next block to look at, first tile in it
  long left;       // tiles of the range not yet handed out
};
__device__ __forceinline__ bool next_seg(const DecodeParams& P, SegIter& it, Seg& s) {
  while (it.left > 0 && it.b < P.num_blocks) {
    const BlockKeys k = block_keys(P, it.b);
    if (it.t < k.nt) {
      s.b = it.b;
      s.t0 = it.t;
      s.n = (int)min((long)(k.nt - it.t), it.left);
      s.k = k;
      it.left -= s.n;
      ++it.b;
      it.t = 0;
      return true;
    }
    ++it.b;
    it.t = 0;
  }
  return false;
}
// The segment's last tile ends its block and holds keys past kv_len.
__device__ __forceinline__ bool seg_ragged_end(const Seg& s) {
  return s.t0 + s.n == s.k.nt && (s.k.kvl - s.k.j_lo) % KT != 0;
}

// Block-wide exclusive scan over the CTA's threads (every thread calls).
__device__ __forceinline__ int block_excl_scan(int v, int* sc, int tid, int* total) {
  const int lane = tid % 32, warp = tid / 32;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) sc[warp] = x;
  __syncthreads();
  int base = 0, tot = 0;
#pragma unroll
  for (int w = 0; w < THREADS / 32; ++w) {
    const int s = sc[w];
    base += w < warp ? s : 0;
    tot += s;
  }
  __syncthreads();
  *total = tot;
  return base + x - v;
}

__global__ void __launch_bounds__(THREADS, 1) latent_decode_tc_kernel(const __grid_constant__ DecodeParams P) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  Bars* B = (Bars*)(smem + OFF_BAR);
  float* red = (float*)(smem + OFF_RED);
  int* redi = (int*)red;
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  const int c = blockIdx.x, nb = P.num_blocks;
  const int R = P.T * P.H;                                  // live rows (<= 32)

  if (tid == 0) {
    for (int s = 0; s < NSLOT; ++s) {
      mbar_init(&B->full[s], 1);
      mbar_init(&B->empty[s], 1);
    }
    mbar_init(&B->vready, 1);
    mbar_init(&B->vfix, 1);
    mbar_init(&B->q_full, 1);
    mbar_init(&B->q_empty, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&B->s_full[i], 1);
      mbar_init(&B->p_full[i], 128);
    }
    mbar_init(&B->o_done, 1);
    mbar_init(&B->o_seg, 1);
    mbar_init(&B->drain, 1);
    B->abort = 0;
    fence_mbar_init();
  }
  if (warp == 4) tmem_alloc(&B->tmem_slot, TMEM_COLS);

  // ---- schedule: total tiles U, then the block holding this CTA's first
  // tile (from the same scan when every block has a thread)
  int* sc = redi + RD_SCH;
  long long U = 0;
  int my_nt = 0, my_excl = 0;
  for (int base = 0; base < nb; base += THREADS) {
    const int b = base + tid;
    const int nt = b < nb ? block_keys(P, b).nt : 0;
    int tot;
    const int ex = block_excl_scan(nt, sc, tid, &tot);
    if (base == 0) {
      my_nt = nt;
      my_excl = ex;
    }
    U += tot;
  }
  // the first min(gridDim, U) CTAs take one range each, so none is empty
  const int G = (int)min((long long)gridDim.x, max(U, 1LL));
  const long long u0 = c < G ? U * c / G : U, u1 = c < G ? U * (c + 1) / G : U;
  if (tid == 0) { sc[12] = nb; sc[13] = 0; }
  __syncthreads();
  if (u1 > u0) {
    if (nb <= THREADS) {
      if (my_nt > 0 && u0 >= my_excl && u0 < my_excl + my_nt) {
        sc[12] = tid;
        sc[13] = (int)(u0 - my_excl);
      }
    } else {
      long long run = 0;
      for (int base = 0; base < nb; base += THREADS) {
        const int b = base + tid;
        const int nt = b < nb ? block_keys(P, b).nt : 0;
        int tot;
        const long long excl = run + block_excl_scan(nt, sc, tid, &tot);
        if (nt > 0 && u0 >= excl && u0 < excl + nt) {
          sc[12] = b;
          sc[13] = (int)(u0 - excl);
        }
        run += tot;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = B->tmem_slot;
  const int b_first = sc[12], t_first = sc[13];
  const long ntiles = (long)(u1 - u0);
  if (tid == 0) pdl_trigger();
  // Each role looks up what it needs from the descriptor (lengths, windows,
  // positions, page rows: inputs of the call, not outputs of the kernels
  // before this one) and then waits for the previous kernel before it
  // touches Q_abs, the cache or the workspace.

  if (warp == 4) {
    if (lane == 0 && ntiles > 0) {
      // ---- MMA issuer ----
      // One thread's issue rate is set by the instructions between its MMAs,
      // so every shared-memory descriptor is a base computed once plus a
      // constant offset (16-byte units) and the ring position advances by
      // increments.
      const uint32_t id_s = idesc_f16(128, NR, false);                 // K-major A and B
      const uint32_t id_o = idesc_f16(128, NR, false) | (1u << 15);    // A (V^T) MN-major
      const uint64_t dK = smem_desc_sw128(smem + OFF_RING);
      const uint64_t dQ = smem_desc_sw128(smem + OFF_Q);
      const uint64_t dV = smem_desc_sw128_mn(smem + OFF_RING, KV_CH_BYTES);
      const uint64_t dP = smem_desc_sw128(smem + OFF_P);
      constexpr uint32_t U_SLOT = SLOT_BYTES / 16, U_CH = KV_CH_BYTES / 16, U_Q = Q_CH_BYTES / 16;
      constexpr uint32_t U_P = P_CH_BYTES / 16, U_PB = P_BYTES / 16, U_KSTEP = 16 * 128 / 16;
      // the four 16-dim steps of one 64-dim chunk of S^T
      auto s4 = [&](uint32_t d, uint64_t a, uint64_t b, uint32_t acc0) {
        mma_f16(d, a, b, id_s, acc0);
        mma_f16(d, a + 2, b + 2, id_s, 1u);
        mma_f16(d, a + 4, b + 4, id_s, 1u);
        mma_f16(d, a + 6, b + 6, id_s, 1u);
      };
      // the eight 16-key steps of one 128-dim value group of O^T
      auto o8 = [&](uint32_t d, uint64_t a, uint64_t p, uint32_t acc0) {
        mma_f16(d, a, p, id_o, acc0);
        mma_f16(d, a + U_KSTEP, p + 2, id_o, 1u);
        mma_f16(d, a + 2 * U_KSTEP, p + 4, id_o, 1u);
        mma_f16(d, a + 3 * U_KSTEP, p + 6, id_o, 1u);
        mma_f16(d, a + 4 * U_KSTEP, p + U_P, id_o, 1u);
        mma_f16(d, a + 5 * U_KSTEP, p + U_P + 2, id_o, 1u);
        mma_f16(d, a + 6 * U_KSTEP, p + U_P + 4, id_o, 1u);
        mma_f16(d, a + 7 * U_KSTEP, p + U_P + 6, id_o, 1u);
      };
      SegIter it{b_first, t_first, ntiles};
      Seg s, nx;
      uint32_t slot = 0, sph = 0;             // ring slot of the next item, its fill parity
      uint32_t g = 0, kseg = 0, nfix = 0;
      bool ok = true, have = next_seg(P, it, s);
      pdl_wait();
      auto advance = [&]() {
        if (++slot == NSLOT) {
          slot = 0;
          sph ^= 1;
        }
      };
      // This thread is the ring's one consumer: every earlier item is
      // consumed, so the next n items are at most one phase ahead and can be
      // probed together (one probe latency instead of one per item when they
      // have all landed, the usual case).
      auto ready = [&](int n) {
        uint32_t sl = slot, ph = sph;
        bool r = true;
#pragma unroll
        for (int q = 0; q < K_ITEMS; ++q) {
          if (q < n) r &= mbar_test_wait(&B->full[sl], ph);
          if (++sl == NSLOT) {
            sl = 0;
            ph ^= 1;
          }
        }
        return r;
      };
      auto wait_item = [&]() {
        if (!wait_bar(B, &B->full[slot], sph, P.status)) return false;
        tc_fence_after();
        return true;
      };
      while (ok && have) {
        const bool have_next = next_seg(P, it, nx);     // looked up ahead of its use
        if (!(ok = wait_bar(B, &B->q_full, kseg & 1, P.status))) break;
        tc_fence_after();
        const uint32_t ob = tmem + TM_O + 128 * (kseg & 1);
        const bool ragged = seg_ragged_end(s);
        for (int t = 0; t <= s.n && ok; ++t) {
          if (t < s.n) {
            // S^T(g + t) into its buffer: pairs 0-1 .. 6-7, then the rope chunk
            const uint32_t ts = tmem + TM_S + 32 * ((g + t) & 1);
            const bool all_in = ready(K_ITEMS);
            if (all_in) tc_fence_after();
            for (int q = 0; q < 4; ++q) {
              if (!all_in && !(ok = wait_item())) break;
              const uint64_t a = dK + slot * U_SLOT, b = dQ + 2 * q * U_Q;
              s4(ts, a, b, q == 0 ? 0u : 1u);
              s4(ts, a + U_CH, b + U_Q, 1u);
              mma_commit(&B->empty[slot]);
              advance();
            }
            if (!ok) break;
            if (!all_in && !(ok = wait_item())) break;
            s4(ts, dK + slot * U_SLOT, dQ + 8 * U_Q, 1u);
            mma_commit(&B->empty[slot]);
            advance();
            mma_commit(&B->s_full[(g + t) & 1]);
            if (t == s.n - 1) mma_commit(&B->q_empty);
          }
          if (t >= 1) {
            // O^T(g + t - 1) once its P is written
            const uint32_t gg = g + t - 1;
            const bool ragged_tile = ragged && t == s.n;
            bool all_in = !ragged_tile && (mbar_test_wait(&B->p_full[gg & 1], (gg >> 1) & 1) & ready(V_ITEMS));
            if (!all_in && !(ok = wait_bar(B, &B->p_full[gg & 1], (gg >> 1) & 1, P.status))) break;
            tc_fence_after();
            if (ragged_tile) {
              // the block's last tile: hand its landed value items to warp 7
              uint32_t sl = slot, ph = sph;
              for (int q = 0; q < V_ITEMS && ok; ++q) {
                ok = wait_bar(B, &B->full[sl], ph, P.status);
                if (++sl == NSLOT) {
                  sl = 0;
                  ph ^= 1;
                }
              }
              if (!ok) break;
              mbar_arrive(&B->vready);
              if (!(ok = wait_bar(B, &B->vfix, nfix & 1, P.status))) break;
              ++nfix;
              tc_fence_after();
              all_in = true;
            }
            const uint64_t pb = dP + (gg & 1) * U_PB;
            const uint32_t acc0 = t == 1 ? 0u : 1u;
            for (int q = 0; q < V_ITEMS; ++q) {
              if (!all_in && !(ok = wait_item())) break;
              o8(ob + 32 * q, dV + slot * U_SLOT, pb, acc0);
              mma_commit(&B->empty[slot]);
              advance();
            }
            if (!ok) break;
            mma_commit(&B->o_done);
            if (t == s.n) mma_commit(&B->o_seg);
          }
        }
        g += s.n;
        ++kseg;
        s = nx;
        have = have_next;
      }
      mma_commit(&B->drain);
      mbar_wait(&B->drain, 0, P.status);
    }
  } else if (warp == 5 || warp == 6) {
    if (lane == 0 && ntiles > 0) {
      // ---- ring copies: this warp fills the slots s with s % 2 == p ----
      const int p = warp - 5;
      const int ps = P.page_size, past_end = P.num_pages * ps;
      prefetch_tmap(&P.tmK1);
      prefetch_tmap(&P.tmK2);
      const uint64_t evict_first = l2_policy_evict_first();
      SegIter it{b_first, t_first, ntiles};
      Seg s;
      uint32_t item = 0;
      uint32_t last_use = 0;          // bit sl: slot sl was filled; bit 8 + sl: the phase of its last fill
      bool ok = true, waited = false;
      auto load = [&](int y0, int q, bool value) {
        const uint32_t slot = item % NSLOT, ph = (item / NSLOT) & 1;
        if ((int)(slot % 2) == p) {
          if (!(ok = wait_bar(B, &B->empty[slot], ph ^ 1, P.status))) return;
          uint8_t* dst = smem + OFF_RING + slot * SLOT_BYTES;
          if (!value && q == 4) {
            mbar_arrive_expect_tx(&B->full[slot], KV_CH_BYTES);
            tma_load_3d(dst, &P.tmK1, &B->full[slot], 8 * DCH, y0, 0);
          } else if (!value) {
            mbar_arrive_expect_tx(&B->full[slot], SLOT_BYTES);
            tma_load_3d(dst, &P.tmK2, &B->full[slot], 0, y0, 2 * q);
          } else {
            // the value pass is the last touch of these lines: first out of L2
            mbar_arrive_expect_tx(&B->full[slot], SLOT_BYTES);
            tma_load_3d_hint(dst, &P.tmK2, &B->full[slot], 0, y0, 2 * q, evict_first);
          }
          last_use = (last_use & ~(0x101u << slot)) | (1u << slot) | (ph << (8 + slot));
        }
        ++item;
      };
      bool have = next_seg(P, it, s);
      while (ok && have) {
        // first cache row of tile t of the segment (past_end for an invalid page: zeros)
        auto tile_row = [&](int t) {
          const int j0 = s.k.j_lo + (s.t0 + t) * KT;
          const int pg = P.block_table[(long)s.b * P.max_pages + j0 / ps];
          if (pg < 0 || pg >= P.num_pages) {
            set_status(P.status, MLA_DEV_BAD_PAGE);
            return past_end;
          }
          return pg * ps + j0 % ps;
        };
        int y_prev = 0, y = tile_row(0);
        for (int t = 0; t <= s.n && ok; ++t) {
          const int y_next = t + 1 < s.n ? tile_row(t + 1) : 0;   // one tile ahead
          if (!waited) {
            pdl_wait();
            waited = true;
          }
          if (t < s.n)
            for (int q = 0; q < K_ITEMS && ok; ++q) load(y, q, false);
          if (t >= 1)
            for (int q = 0; q < V_ITEMS && ok; ++q) load(y_prev, q, true);
          y_prev = y;
          y = y_next;
        }
        have = next_seg(P, it, s);
      }
      // the copies in flight land before the CTA exits
      for (int sl = 0; sl < NSLOT; ++sl)
        if (last_use & (1u << sl)) mbar_wait(&B->full[sl], (last_use >> (8 + sl)) & 1, P.status);
    }
  } else if (warp == 7) {
    if (ntiles > 0) {
      // ---- Q of each segment; value rows past kv_len zeroed ----
      SegIter it{b_first, t_first, ntiles};
      Seg cur, nxt;
      bool have = next_seg(P, it, cur), ok = true;
      uint32_t item_base = 0, kseg = 0, nq = 0, nfix = 0;
      pdl_wait();
      if (lane == 0) {
        prefetch_tmap(&P.tmQ);
        mbar_arrive_expect_tx(&B->q_full, NCH * Q_CH_BYTES);
        tma_load_3d(smem + OFF_Q, &P.tmQ, &B->q_full, 0, cur.b * R, 0);
      }
      ++nq;
      while (have && ok) {
        const bool have_next = next_seg(P, it, nxt);
        if (have_next) {
          // Q of the next segment once every S^T of this one is done
          if (lane == 0) {
            ok = wait_bar(B, &B->q_empty, kseg & 1, P.status);
            if (ok) {
              mbar_arrive_expect_tx(&B->q_full, NCH * Q_CH_BYTES);
              tma_load_3d(smem + OFF_Q, &P.tmQ, &B->q_full, 0, nxt.b * R, 0);
            }
          }
          ok = __shfl_sync(0xffffffffu, ok, 0);
          if (ok) ++nq;
        }
        if (ok && seg_ragged_end(cur)) {
          const int j0 = cur.k.j_lo + (cur.t0 + cur.n - 1) * KT;
          const int valid = cur.k.kvl - j0;                   // 1 .. 127 live rows
          const int units = (KT - valid) * 16;                // 16-byte units past kv_len, per item
          ok = __all_sync(0xffffffffu, wait_bar(B, &B->vready, nfix & 1, P.status));
          if (ok) {
            for (int q = 0; q < V_ITEMS; ++q) {
              const uint32_t slot = (item_base + 9 * cur.n - V_ITEMS + q) % NSLOT;
              uint8_t* sp = smem + OFF_RING + slot * SLOT_BYTES;
              for (int i = lane; i < units; i += 32) {
                const int row = valid + i / 16, part = i % 16;
                *reinterpret_cast<uint4*>(sp + (part / 8) * KV_CH_BYTES + row * 128 + (part % 8) * 16) =
                    make_uint4(0, 0, 0, 0);
              }
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&B->vfix);
            ++nfix;
          }
        }
        item_base += 9 * cur.n;
        cur = nxt;
        have = have_next;
        ++kseg;
      }
      if (lane == 0) mbar_wait(&B->q_full, (nq - 1) & 1, P.status);
    }
  } else {
    // ---- softmax warps: thread k = key k of the tile (TMEM lane k) ----
    const int k = tid;
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    float* wpart = red + RD_WPART;
    float* m_s = red + RD_M;
    float* al_s = red + RD_ALPHA;
    float* il_s = red + RD_INVL;
    int* rlo = redi + RD_LO;
    int* rhi = redi + RD_HI;
    // Before their first global write these warps wait for the previous
    // kernel (the workspace may still be read by it); the first CTA then
    // records each block's segment range for the merge.
    bool waited = false;
    auto first_write = [&]() {
      if (waited) return;
      waited = true;
      pdl_wait();
      if (c == 0) {
        // each block's segments for the merge (first CTA, count); invalid
        // lengths and windows reported once
        long long run = 0;
        for (int base = 0; base < nb; base += 128) {
          const int b = base + k;
          BlockKeys bk{};
          if (b < nb) {
            bk = block_keys(P, b);
            if (bk.bad_len) set_status(P.status, MLA_DEV_BAD_LENGTH);
            if (bk.bad_win) set_status(P.status, MLA_DEV_BAD_WINDOW);
          }
          int x = bk.nt;
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
          }
          if (lane == 31) redi[RD_WPART + warp] = x;
          softmax_sync();
          int wb = 0, tot = 0;
#pragma unroll
          for (int w = 0; w < 4; ++w) {
            const int sv = redi[RD_WPART + w];
            wb += w < warp ? sv : 0;
            tot += sv;
          }
          softmax_sync();
          const long long excl = run + wb + x - bk.nt;
          if (b < nb) {
            const int f = bk.nt ? cta_of(excl, U, G) : 0;
            const int l = bk.nt ? cta_of(excl + bk.nt - 1, U, G) : -1;
            P.meta[2 * (long)b] = f;
            P.meta[2 * (long)b + 1] = l - f + 1;
          }
          run += tot;
        }
      }
    };
    SegIter it{b_first, t_first, ntiles};
    Seg s, nx;
    uint32_t g = 0, kseg = 0;
    long long u_seg = u0;                     // global index of the segment's first tile
    bool have = next_seg(P, it, s);
    while (have) {
      const bool have_next = next_seg(P, it, nx);
      const int b = s.b;
      const long slot = (long)b + c;
      const int k_begin = s.k.j_lo + s.t0 * KT;              // first key of the segment
      const int k_end = min(s.k.kvl, k_begin + s.n * KT);
      const uint32_t ob = tmem + TM_O + 128 * (kseg & 1);
      softmax_sync();                          // the previous segment's epilogue is done with the rows
      if (k < NR) {
        int lo = 0, hi = 0;
        if (k < R) {
          const long m = (long)b * P.T + k / P.H;
          const int pq = P.positions[m];
          const bool qv = P.q_visible ? P.q_visible[m] != 0 : true;
          lo = s.k.W > 0 ? max(0, pq - s.k.W + 1) : 0;
          hi = qv ? s.k.kvl : 0;
        }
        rlo[k] = lo;
        rhi[k] = hi;
      }
      softmax_sync();
      float lrow[NR];
#pragma unroll
      for (int r = 0; r < NR; ++r) lrow[r] = 0.f;
      for (int t = 0; t < s.n; ++t) {
        const uint32_t gg = g + t;
        const int j = k_begin + t * KT + k;   // this thread's key
        float sv[NR];
        wait_bar(B, &B->s_full[gg & 1], (gg >> 1) & 1, P.status);
        tc_fence_after();
        tmem_ld32_nowait(tmem + TM_S + 32 * (gg & 1) + lane_base, sv);
        tmem_ld_wait();
        tmem_reg_fence32(sv);
        // mask by logical position: row r sees keys [lo_r, hi_r)
#pragma unroll
        for (int r = 0; r < NR; r += 4) {
          const int4 lo4 = *reinterpret_cast<const int4*>(rlo + r), hi4 = *reinterpret_cast<const int4*>(rhi + r);
          sv[r] = (j >= lo4.x && j < hi4.x) ? sv[r] : -INFINITY;
          sv[r + 1] = (j >= lo4.y && j < hi4.y) ? sv[r + 1] : -INFINITY;
          sv[r + 2] = (j >= lo4.z && j < hi4.z) ? sv[r + 2] : -INFINITY;
          sv[r + 3] = (j >= lo4.w && j < hi4.w) ? sv[r + 3] : -INFINITY;
        }
        float x[NR];
#pragma unroll
        for (int r = 0; r < NR; ++r) x[r] = sv[r];
        wpart[warp * 32 + lane] = warp_transpose_reduce<true>(x, lane);   // lane l: max of row l
        softmax_sync();
        if (warp == 0) {
          // row `lane`: running max (exp2 domain) and the factor for what is accumulated
          const float cm = fmaxf(fmaxf(wpart[lane], wpart[32 + lane]), fmaxf(wpart[64 + lane], wpart[96 + lane]));
          const float tm = cm * P.scale_log2, m_old = t == 0 ? -INFINITY : m_s[lane];
          const bool grow = tm > m_old + RESCALE_LOG2;
          const float m_new = grow ? tm : m_old;
          const float alpha = (grow && m_old != -INFINITY) ? exp2f(m_old - m_new) : 1.f;
          m_s[lane] = m_new;
          al_s[lane] = alpha;
          const bool any = __any_sync(0xffffffffu, alpha != 1.f);
          if (lane == 0) redi[RD_FLAG] = any;
        }
        softmax_sync();
        const bool rescale = redi[RD_FLAG] != 0;
        // O^T(gg - 1) is issued after S^T(gg) (and O^T(gg) only after this
        // tile's P): a row that grew waits for it, then rescales
        if (rescale && t > 0) {
          wait_bar(B, &B->o_done, (gg - 1) & 1, P.status);
          tc_fence_after();
#pragma unroll 1
          for (int q = 0; q < 4; ++q) {
            float o[NR];
            tmem_ld32_nowait(ob + 32 * q + lane_base, o);
            tmem_ld_wait();
            tmem_reg_fence32(o);
#pragma unroll
            for (int r = 0; r < NR; r += 4) {
              const float4 av = *reinterpret_cast<const float4*>(al_s + r);
              o[r] *= av.x; o[r + 1] *= av.y; o[r + 2] *= av.z; o[r + 3] *= av.w;
            }
            tmem_st32(ob + 32 * q + lane_base, o);
          }
        }
        // P[r][k] (bf16) into the swizzled K-major tile: 16-byte unit (k % 64) / 8
        // of row r sits at unit ((k % 64) / 8) ^ (r % 8); each row's max and
        // factor read four rows at a time (short live ranges)
        uint8_t* pchunk = smem + OFF_P + (gg & 1) * P_BYTES + (k / 64) * P_CH_BYTES;
        const int kk = k % 64;
#pragma unroll
        for (int r4 = 0; r4 < NR; r4 += 4) {
          const float4 mv = *reinterpret_cast<const float4*>(m_s + r4);
          const float4 av = *reinterpret_cast<const float4*>(al_s + r4);
          const float mr[4] = {mv.x, mv.y, mv.z, mv.w}, ar[4] = {av.x, av.y, av.z, av.w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int r = r4 + i;
            const float m0 = mr[i] == -INFINITY ? 0.f : mr[i];
            const float p = fast_exp2(fmaf(sv[r], P.scale_log2, -m0));
            lrow[r] = fmaf(lrow[r], ar[i], p);
            *reinterpret_cast<__nv_bfloat16*>(pchunk + r * 128 + (((kk >> 3) ^ (r & 7)) << 4) + (kk & 7) * 2) =
                __float2bfloat16_rn(p);
          }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(&B->p_full[gg & 1]);
      }
      // ---- epilogue of the segment: row sums, then either the block's final
      // output (the block lies in this CTA alone) or a normalised partial
      first_write();
      const long long S_b = u_seg - s.t0;                     // the block's first tile, global order
      const int fb = cta_of(S_b, U, G), nseg = cta_of(S_b + s.k.nt - 1, U, G) - fb + 1;
      const bool direct = nseg == 1;
      float x[NR];
#pragma unroll
      for (int r = 0; r < NR; ++r) x[r] = lrow[r];
      wpart[warp * 32 + lane] = warp_transpose_reduce<false>(x, lane);
      softmax_sync();
      if (warp == 0) {
        const float l = (wpart[lane] + wpart[32 + lane]) + (wpart[64 + lane] + wpart[96 + lane]);
        il_s[lane] = l > 0.f ? 1.f / l : 0.f;
        const float l2 = l > 0.f ? m_s[lane] + log2f(l) : -INFINITY;
        if (!direct)
          P.part_lse[slot * NR + lane] = l2;
        else if (P.lse && lane < R)
          P.lse[(long)b * R + lane] = l2 == -INFINITY ? -INFINITY : l2 * 0.6931471805599453f;
      }
      softmax_sync();
      float il[NR];
#pragma unroll
      for (int r = 0; r < NR; r += 4) {
        const float4 v = *reinterpret_cast<const float4*>(il_s + r);
        il[r] = v.x; il[r + 1] = v.y; il[r + 2] = v.z; il[r + 3] = v.w;
      }
      wait_bar(B, &B->o_seg, kseg & 1, P.status);
      tc_fence_after();
      // thread k holds value dim 128 q + k of every row (a row nothing was
      // visible to stays +0)
#pragma unroll 1
      for (int q = 0; q < 4; ++q) {
        float o[NR];
        tmem_ld32_nowait(ob + 32 * q + lane_base, o);
        tmem_ld_wait();
        tmem_reg_fence32(o);
#pragma unroll
        for (int r = 0; r < NR; ++r) o[r] = il[r] > 0.f ? o[r] * il[r] : 0.f;
        if (direct) {
#pragma unroll
          for (int r = 0; r < NR; ++r)
            if (r < R) P.o_lat[((long)b * R + r) * 512 + 128 * q + k] = __float2half_rn(o[r]);
        } else {
          // row-major, so that a warp's store is one 128-byte line; kept in
          // L2 for the merge (the cache stream would push them out)
          float* dst = P.part + slot * NR * 512 + 128 * q + k;
          const uint64_t keep = l2_policy_evict_last();
#pragma unroll
          for (int r = 0; r < NR; ++r) st_global_hint(dst + r * 512, o[r], keep);
        }
      }
      if (k < P.T) {   // visibility of token k over this segment's keys (one interval)
        const int lo = max(rlo[k * P.H], k_begin), hi = min(rhi[k * P.H], k_end);
        int* vs = direct ? (P.vis_stats ? P.vis_stats + ((long)b * P.T + k) * 3 : nullptr)
                         : P.part_vis + (slot * P.T + k) * 3;
        if (vs) {
          vs[0] = hi > lo ? hi - lo : 0;
          vs[1] = hi > lo ? lo : -1;
          vs[2] = hi > lo ? hi - 1 : -1;
        }
      }
      u_seg += s.n;
      tc_fence_before();
      g += s.n;
      ++kseg;
      s = nx;
      have = have_next;
    }
    first_write();
  }
  pdl_wait();        // (a no-op for the threads that waited already)
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 4) tmem_dealloc(tmem, TMEM_COLS);
}

// Grid (block, quarter of the value dims): the segments' partials of each
// row combined by log-sum-exp in CTA order; a row no segment saw stays
// exactly zero, a block with no keys is all zero, a block held by one CTA
// was written directly by it.  Thread i handles value dims 128 * quarter +
// 4 (i % 32) .. + 3 of rows i / 32 + 8 j (j < 4): a warp's load of one
// row is 512 contiguous bytes; MERGE_LOADS segments' rows are in flight at
// once.  Eight threads derive the weights of each row.
constexpr int MERGE_THREADS = 256, MERGE_SPLIT = 4, MERGE_LOADS = 4;
constexpr int MERGE_SMEM_MAX = 200 * (NR + 3 * NR) * 4;   // up to 200 segments of 32 one-token blocks
__global__ void __launch_bounds__(MERGE_THREADS, 2) decode_merge_kernel(const __grid_constant__ DecodeParams P) {
  extern __shared__ float w_s[];              // [segments][32] log2-sum-exps then weights; [segments][T][3] visibility
  __shared__ float lse_s[NR];
  const int b = blockIdx.x, part = blockIdx.y, tid = threadIdx.x;
  const int R = P.T * P.H;
  const int f = P.meta[2 * (long)b], cnt = P.meta[2 * (long)b + 1];
  if (cnt == 1) return;
  const long slot0 = (long)b + f;
  const bool lead = part == 0;
  int* vis_s = reinterpret_cast<int*>(w_s + cnt * NR);
  for (int i = tid; i < cnt * NR; i += MERGE_THREADS) w_s[i] = P.part_lse[slot0 * NR + i];
  if (lead && P.vis_stats)
    for (int i = tid; i < cnt * P.T * 3; i += MERGE_THREADS) vis_s[i] = P.part_vis[slot0 * P.T * 3 + i];
  __syncthreads();
  {
    // row tid / 8, segments tid % 8 + 8 j
    const int r = tid / 8, sl = tid % 8;
    float mx = -INFINITY;
    for (int s = sl; s < cnt; s += 8) mx = fmaxf(mx, w_s[s * NR + r]);
#pragma unroll
    for (int o = 4; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    float den = 0.f;
    for (int s = sl; s < cnt; s += 8) {
      const float l = w_s[s * NR + r];
      const float w = (mx == -INFINITY || l == -INFINITY) ? 0.f : exp2f(l - mx);
      w_s[s * NR + r] = w;
      den += w;
    }
#pragma unroll
    for (int o = 4; o > 0; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
    const float inv = den > 0.f ? 1.f / den : 0.f;
    for (int s = sl; s < cnt; s += 8) w_s[s * NR + r] *= inv;
    if (sl == 0) lse_s[r] = den > 0.f ? mx + log2f(den) : -INFINITY;
  }
  __syncthreads();
  const int d = 128 * part + 4 * (tid % 32), r0 = tid / 32;
  float acc[4][4];
#pragma unroll
  for (int j = 0; j < 4; ++j)
#pragma unroll
    for (int e = 0; e < 4; ++e) acc[j][e] = 0.f;
  for (int s0 = 0; s0 < cnt; s0 += MERGE_LOADS) {
    float4 v[MERGE_LOADS][4];
#pragma unroll
    for (int i = 0; i < MERGE_LOADS; ++i)
      if (s0 + i < cnt) {
        const float* src = P.part + ((slot0 + s0 + i) * NR + r0) * 512 + d;
#pragma unroll
        for (int j = 0; j < 4; ++j) v[i][j] = *reinterpret_cast<const float4*>(src + 8 * j * 512);
      }
#pragma unroll
    for (int i = 0; i < MERGE_LOADS; ++i)
      if (s0 + i < cnt) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float w = w_s[(s0 + i) * NR + r0 + 8 * j];
          acc[j][0] = fmaf(w, v[i][j].x, acc[j][0]);
          acc[j][1] = fmaf(w, v[i][j].y, acc[j][1]);
          acc[j][2] = fmaf(w, v[i][j].z, acc[j][2]);
          acc[j][3] = fmaf(w, v[i][j].w, acc[j][3]);
        }
      }
  }
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int r = r0 + 8 * j;
    if (r < R) {
      const __half2 lo = __floats2half2_rn(acc[j][0], acc[j][1]), hi = __floats2half2_rn(acc[j][2], acc[j][3]);
      uint2 u;
      u.x = *reinterpret_cast<const uint32_t*>(&lo);
      u.y = *reinterpret_cast<const uint32_t*>(&hi);
      *reinterpret_cast<uint2*>(P.o_lat + ((long)b * R + r) * 512 + d) = u;
    }
  }
  if (lead && tid < R && P.lse) {
    const float l2 = lse_s[tid];
    P.lse[(long)b * R + tid] = l2 == -INFINITY ? -INFINITY : l2 * 0.6931471805599453f;
  }
  // visibility statistics of each token
  if (lead && tid < P.T && P.vis_stats) {
    int n = 0, first = -1, last = -1;
    for (int s = 0; s < cnt; ++s) {
      const int* vs = vis_s + (s * P.T + tid) * 3;
      if (vs[0] > 0) {
        first = n ? min(first, vs[1]) : vs[1];
        last = max(last, vs[2]);
        n += vs[0];
      }
    }
    const long m = (long)b * P.T + tid;
    P.vis_stats[m * 3 + 0] = n;
    P.vis_stats[m * 3 + 1] = n ? first : -1;
    P.vis_stats[m * 3 + 2] = n ? last : -1;
  }
}

// Workspace pieces: partial slots block + CTA < num_blocks + grid.
size_t ws_layout(long num_blocks, int grid, int T, size_t* off_lse, size_t* off_vis, size_t* off_meta) {
  const long slots = num_blocks + grid;
  size_t o = align256((size_t)slots * NR * 512 * 4);
  *off_lse = o;
  o += align256((size_t)slots * NR * 4);
  *off_vis = o;
  o += align256((size_t)slots * T * 3 * 4);
  *off_meta = o;
  o += align256((size_t)num_blocks * 2 * 4);
  return o;
}

}  // namespace

bool decode_applies(const mla_handle* h, int block_len) {
  const Layout& l = h->lay;
  return h->cfg.dtype == MLA_BF16 && l.rkv == 512 && l.dr == 64 && block_len * l.H <= NR &&
         h->cfg.page_size % KT == 0;
}

size_t decode_workspace_bytes(const mla_handle* h, const mla_attn_desc_t& d) {
  size_t a, b, c;
  return ws_layout(d.num_blocks, h->num_sms, d.block_len, &a, &b, &c);
}

size_t decode_workspace_bound(const mla_handle* h, long max_blocks, int max_block_len) {
  size_t a, b, c;
  return ws_layout(max_blocks, h->num_sms, max_block_len, &a, &b, &c);
}

mla_status_t latent_decode(cudaStream_t st, const mla_handle* h, const __nv_bfloat16* q_abs,
                           const __nv_bfloat16* cache, int num_pages, const mla_attn_desc_t& d,
                           const int32_t* positions, __half* o_lat, float* lse, void* workspace,
                           size_t workspace_bytes, bool pdl) {
  const Layout& l = h->lay;
  if (!decode_applies(h, d.block_len))
    return fail(MLA_ERR_UNSUPPORTED, "decode attention: needs block_len * num_heads <= 32, page_size a multiple of 128");
  if (d.num_blocks <= 0) return MLA_OK;
  size_t off_lse, off_vis, off_meta;
  const int G = h->num_sms;
  if ((size_t)G * (NR + 3 * d.block_len) * 4 > (size_t)MERGE_SMEM_MAX)
    return fail(MLA_ERR_UNSUPPORTED, "decode attention: more than 200 SMs");
  const size_t need = ws_layout(d.num_blocks, G, d.block_len, &off_lse, &off_vis, &off_meta);
  if (workspace_bytes < need || (uintptr_t)workspace % 256)
    return fail(MLA_ERR_INVALID_ARG, "decode attention: workspace too small or not 256-byte aligned");
  DecodeParams P;
  const long rows = (long)d.num_blocks * d.block_len * l.H;
  const long slots = (long)num_pages * h->cfg.page_size;
  if (!make_tmap_chunked(&P.tmQ, false, q_abs, rows, l.L, l.L, NR, NCH) ||
      !make_tmap_2d(&P.tmK1, false, cache, slots, l.L, l.L, KT) ||
      !make_tmap_chunked(&P.tmK2, false, cache, slots, l.L, l.L, KT, 2))
    return fail(MLA_ERR_CUDA, "decode attention: cuTensorMapEncodeTiled failed");
  char* ws = (char*)workspace;
  P.part = (float*)ws;
  P.part_lse = (float*)(ws + off_lse);
  P.part_vis = (int*)(ws + off_vis);
  P.meta = (int*)(ws + off_meta);
  P.block_table = d.block_table;
  P.kv_len = d.kv_len;
  P.window = d.window;
  P.q_visible = d.q_visible;
  P.positions = positions;
  P.vis_stats = d.vis_stats;
  P.o_lat = o_lat;
  P.lse = lse;
  P.status = h->status;
  P.num_blocks = d.num_blocks;
  P.max_pages = d.max_pages;
  P.num_pages = num_pages;
  P.page_size = h->cfg.page_size;
  P.T = d.block_len;
  P.H = l.H;
  P.scale_log2 = h->scale * 1.4426950408889634f;
  static std::once_flag once;
  std::call_once(once, [] {
    cudaFuncSetAttribute(latent_decode_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    cudaFuncSetAttribute(decode_merge_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, MERGE_SMEM_MAX);
  });
  Launch L(dim3((unsigned)G), dim3(THREADS), SMEM_BYTES, st, pdl);
  cudaError_t e = cudaLaunchKernelEx(&L.cfg, latent_decode_tc_kernel, P);
  if (e != cudaSuccess) return cuda_fail(e, "decode attention launch");
  // (a programmatic launch of the merge measured slower: it stays a plain one)
  const size_t merge_smem = (size_t)G * (NR + 3 * d.block_len) * 4;
  decode_merge_kernel<<<dim3((unsigned)d.num_blocks, MERGE_SPLIT), MERGE_THREADS, merge_smem, st>>>(P);
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "decode merge launch");
  return MLA_OK;
}

}  // namespace tc
}  // namespace mla
