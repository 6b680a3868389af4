// Expanded-form attention of the MLA draft layer for blocks that share a
// context ("MLA (Multi-Head Latent Attention)" blog, forward_impl: the
// prefill path, forward_mha, whose context keys come from the cache through
// kv_b_proj, _compute_prefill_context, and whose new tokens attend
// themselves, _run_prefill_new_tokens; the two merged by log-sum-exp,
// merge_attn_states).
//
// When thousands of query rows meet one cached context, the absorbed form
// pays 2 * (576 + 512) flop per key and row; the expanded form 2 * (192 +
// 128), after kv_b_proj expands each context latent once into per-head
// k_nope and v.  Here a context's keys and each block's own keys are
// gathered into dense rows, expanded by one GEMM (kv_b_proj, [k_nope | v]
// per head, fp16), and one kernel runs per (up to 128 / block_len blocks of
// a context, head): 128 query rows against the context's key tiles and then
// one more tile holding the blocks' own keys, masked so that each block sees
// its own (a block-diagonal tile).  One online softmax covers both, which is
// the log-sum-exp merge of the two parts done in place.
//
//   S = [q_nope | q_pe] [k_nope | k_pe]^T   (M = 128 rows, N = 128 keys,
//        K = 128 fp16 + 64 bf16: 8 + 4 MMAs)
//   O += P V                                (N = 128 value dims, K = 128
//        keys: 8 MMAs, P fp16 from tensor memory)
// O is 128 fp32 columns and S (with P over it) three buffers of 128: the
// scores of tile t + 1 are computed while the softmax of tile t runs, and
// S(t + 1) waits only for P V of tile t - 2, so the chain softmax -> P V ->
// S -> softmax spans three tiles (two buffers left it on every second tile,
// and the tile period at about half that chain).
//
// Units.  A context's blocks are first ordered full-mask ones before
// windowed ones (a stable partition, expand_units_kernel), and a unit takes
// up to 128 / block_len consecutive blocks of that order: its rows then share
// one mask class, so a windowed unit skips the context tiles below its
// windows and the rows of a warp agree on which keys a tile shows them.
// The unit's query rows and own keys are then loaded block by block (one
// block_len-row box each, at rows that keep the 128-byte swizzle's
// 1024-byte alignment: block_len a multiple of 8 dividing 128); other block
// lengths take consecutive blocks in their given order.
// Keys and values stream through separate two-slot rings: a key slot is
// refilled as soon as its scores are done, so the score chain never waits for
// P V.
//   warps 0-3, 8-11: softmax, two threads per row (64 keys each), half
//                    maxima exchanged through shared memory; epilogue
//                    (thread 0 also issues the unit's Q loads at start)
//   warp 4         : the key tiles (TMA)
//   warp 6         : the value tiles (TMA)
//   warp 5         : tensor-memory allocation, S issue
//   warp 7         : P V issue (two issuing threads: one thread's issue
//                    rate, not the tensor pipe, bounded the tile)
#include "expand_tc.cuh"

#include <mutex>

#include "gemm_tc.cuh"
#include "tc_ptx.cuh"

namespace mla {
namespace tc {
namespace {

constexpr int QROWS = 128, KT = 128;
constexpr int THREADS = 384;
constexpr int CH = 128 * 64 * 2;                 // one 16 KiB chunk: 128 rows x 64 16-bit values
constexpr int OFF_Q = 0;                          // q_nope (2 chunks, fp16), q_pe (bf16)
constexpr int OFF_KR = OFF_Q + 3 * CH;            // key ring, 2 slots: k_nope (2 chunks), k_pe
constexpr int KSLOT = 3 * CH;
constexpr int OFF_VR = OFF_KR + 2 * KSLOT;        // value ring, 2 slots: v (2 chunks)
constexpr int VSLOT = 2 * CH;
constexpr int OFF_BAR = OFF_VR + 2 * VSLOT;
constexpr int OFF_XM = OFF_BAR + 256;             // [2 (tile parity)][2][128] half maxima / sums
constexpr int OFF_RED = OFF_XM + 4 * QROWS * 4;   // [8] per-warp minima of the window starts
constexpr int SMEM_BYTES = 1024 + OFF_RED + 64;
constexpr int NS = 3;                             // S buffers
constexpr uint32_t TMEM_COLS = 512, TM_O = 0, TM_S = 128;   // O 128 columns; S (and P over it) 3 x 128
constexpr float RESCALE_LOG2 = 8.f;
static_assert(SMEM_BYTES <= 232448, "shared memory");

struct Bars {
  uint64_t q_full;
  uint64_t kfull[2], kempty[2]; // key slot landed / read by S (by tile parity)
  uint64_t vfull[2], vempty[2]; // value slot landed / read by P V (by tile parity)
  uint64_t s_full[NS];          // S(t) complete, by t % NS
  uint64_t p_full[NS];          // P(t) in tensor memory (256 arrivals), by t % NS
  uint64_t o_free[NS];          // P(t) V(t) complete, by t % NS
  uint64_t drain, drain_pv;
  uint32_t tmem_slot;
  int abort;
};
static_assert(sizeof(Bars) <= 256, "barrier block");

struct ExpParams {
  CUtensorMap tmQn, tmQp, tmKV, tmKp;       // 128-row boxes (Q of a unit, context key tiles)
  CUtensorMap tmQnT, tmQpT, tmKVT, tmKpT;   // block_len-row boxes, one chunk (grouped units)
  const int32_t* perm;     // [num_blocks]: each context's blocks, full-mask first (NULL: given order)
  const int32_t* ncls;     // [num_ctx][2]: full-mask and windowed block counts
  const int32_t* positions;
  const int32_t* kv_len;
  const int32_t* window;
  const uint8_t* q_visible;
  int32_t* vis_stats;
  const int32_t* ctx_len;
  const int32_t* ctx_start;
  const float* gate;
  long ld_gate;
  __half* o;
  uint32_t* status;
  int num_ctx, ctx_rows, T, H, bpu, rows, M;
  float scale_log2;
};

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
// the two threads of a row sit in warps w and w + 8: each such pair of
// warps synchronises on its own named barrier (4 + w % 4), so the four pairs
// do not wait for one another
__device__ __forceinline__ void pair_sync(int warp) {
  asm volatile("bar.sync %0, 64;" ::"r"(4 + (warp & 3)) : "memory");
}
__device__ __forceinline__ float max3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
// (x0, x1) = (x0 * a - b, x1 * a - b) and (s0, s1) += (x0, x1): paired fp32
// operations, each rounded as its scalar form
__device__ __forceinline__ void fms2(float& x0, float& x1, float a, float nb) {
  uint64_t x, y, c;
  asm("mov.b64 %0, {%1, %2};" : "=l"(x) : "f"(x0), "f"(x1));
  asm("mov.b64 %0, {%1, %1};" : "=l"(y) : "f"(a));
  asm("mov.b64 %0, {%1, %1};" : "=l"(c) : "f"(nb));
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(x) : "l"(x), "l"(y), "l"(c));
  asm("mov.b64 {%0, %1}, %2;" : "=f"(x0), "=f"(x1) : "l"(x));
}
__device__ __forceinline__ void add2(float& s0, float& s1, float x0, float x1) {
  uint64_t a, b;
  asm("mov.b64 %0, {%1, %2};" : "=l"(a) : "f"(s0), "f"(s1));
  asm("mov.b64 %0, {%1, %2};" : "=l"(b) : "f"(x0), "f"(x1));
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(a) : "l"(a), "l"(b));
  asm("mov.b64 {%0, %1}, %2;" : "=f"(s0), "=f"(s1) : "l"(a));
}

// Unit u: entries pstart .. pstart + nbu - 1 (at most bpu) of the block
// order (perm, or the given order) of context c, whose ctx_len keys start at
// row coff of the gathered rows.  With perm, a unit never mixes the
// context's full-mask and windowed blocks.  False past the last unit.
// Called by whole warps: lane l reads context base + l's counts, and the
// unit and key offsets are scans over the lanes (one round of loads for up
// to 32 contexts).
__device__ __forceinline__ bool unit_of(const ExpParams& P, int u, int& c, int& pstart, int& nbu,
                                        int& coff, int& ctx_len) {
  const int lane = threadIdx.x & 31;
  int acc = 0, kacc = 0;
  for (int base = 0; base < P.num_ctx; base += 32) {
    const int cc = base + lane;
    int s = 0, n0 = 0, n1 = 0, len = 0;
    if (cc < P.num_ctx) {
      s = P.ctx_start[cc];
      const int e = P.ctx_start[cc + 1];
      n0 = P.perm ? P.ncls[2 * cc] : max(e - s, 0);
      n1 = P.perm ? P.ncls[2 * cc + 1] : 0;
      len = P.ctx_len[cc];
    }
    const int u0 = (n0 + P.bpu - 1) / P.bpu, nu = u0 + (n1 + P.bpu - 1) / P.bpu;
    int x = nu, y = len;                          // inclusive scans over the lanes
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int xs = __shfl_up_sync(0xffffffffu, x, o), ys = __shfl_up_sync(0xffffffffu, y, o);
      if (lane >= o) {
        x += xs;
        y += ys;
      }
    }
    const unsigned hit = __ballot_sync(0xffffffffu, cc < P.num_ctx && acc + x > u);
    if (hit) {
      const int l = __ffs(hit) - 1;
      const int k = u - acc - __shfl_sync(0xffffffffu, x - nu, l);   // unit within the context
      const int cs = __shfl_sync(0xffffffffu, s, l), cu0 = __shfl_sync(0xffffffffu, u0, l);
      const int cn0 = __shfl_sync(0xffffffffu, n0, l), cn1 = __shfl_sync(0xffffffffu, n1, l);
      c = base + l;
      coff = kacc + __shfl_sync(0xffffffffu, y - len, l);
      ctx_len = __shfl_sync(0xffffffffu, len, l);
      if (k < cu0) {
        pstart = cs + k * P.bpu;
        nbu = min(P.bpu, cn0 - k * P.bpu);
      } else {
        pstart = cs + cn0 + (k - cu0) * P.bpu;
        nbu = min(P.bpu, cn1 - (k - cu0) * P.bpu);
      }
      return true;
    }
    acc += __shfl_sync(0xffffffffu, x, 31);
    kacc += __shfl_sync(0xffffffffu, y, 31);
  }
  return false;
}
__device__ __forceinline__ int unit_block(const ExpParams& P, int pstart, int i) {
  return P.perm ? P.perm[pstart + i] : pstart + i;
}

__global__ void __launch_bounds__(THREADS, 1) expand_attn_kernel(const __grid_constant__ ExpParams P) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  Bars* B = (Bars*)(smem + OFF_BAR);
  float* xm = (float*)(smem + OFF_XM);
  int* red = (int*)(smem + OFF_RED);
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  const int h = blockIdx.y;
  int c, pstart, nbu, coff, ctx_len;
  pdl_wait();                  // the block order comes from the kernel before this one
  if (!unit_of(P, blockIdx.x, c, pstart, nbu, coff, ctx_len)) return;   // the grid is an upper bound
  const int T = P.T, nrows = nbu * T;
  const bool grouped = P.perm != nullptr;
  const long m0 = (long)pstart * T;                             // (contiguous units) first query row
  const long own0 = (long)P.ctx_rows + m0;                      // (contiguous units) first own-key row
  const int slots = QROWS / T;                                  // block_len-row groups of a tile (grouped)

  if (tid == 0) {
    mbar_init(&B->q_full, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&B->kfull[i], 1);
      mbar_init(&B->kempty[i], 1);
      mbar_init(&B->vfull[i], 1);
      mbar_init(&B->vempty[i], 1);
    }
    for (int i = 0; i < NS; ++i) {
      mbar_init(&B->s_full[i], 1);
      mbar_init(&B->p_full[i], 2 * QROWS);
      mbar_init(&B->o_free[i], 1);
    }
    mbar_init(&B->drain, 1);
    mbar_init(&B->drain_pv, 1);
    B->abort = 0;
    fence_mbar_init();
    // the unit's queries, issued before anything else waits: block i's rows
    // at rows i T of the tile (grouped units), the rest past the end (zeros)
    mbar_arrive_expect_tx(&B->q_full, 3 * CH);
    if (!grouped) {
      tma_load_3d(smem + OFF_Q, &P.tmQn, &B->q_full, 0, (int)m0, 2 * h);
      tma_load_3d(smem + OFF_Q + 2 * CH, &P.tmQp, &B->q_full, 0, (int)m0, 9 * h + 8);
    } else {
      int row[16];                                // slots <= 16 (block_len >= 8)
#pragma unroll
      for (int i = 0; i < 16; ++i) row[i] = i < nbu ? P.perm[pstart + i] * T : P.M;
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        if (i < slots) {
          uint8_t* dst = smem + OFF_Q + i * T * 128;
          tma_load_3d(dst, &P.tmQnT, &B->q_full, 0, row[i], 2 * h);
          tma_load_3d(dst + CH, &P.tmQnT, &B->q_full, 0, row[i], 2 * h + 1);
          tma_load_3d(dst + 2 * CH, &P.tmQpT, &B->q_full, 0, row[i], 9 * h + 8);
        }
      }
    }
  }
  if (warp == 5) tmem_alloc(&B->tmem_slot, TMEM_COLS);
  // first context key any row of the unit can see (whole tiles below it are
  // skipped): the least window start over the unit's rows (0 for a full mask)
  int lo_r = 0x7fffffff;
  if (tid < QROWS && tid < nrows) {
    const int b = unit_block(P, pstart, tid / T);
    const int W = P.window ? P.window[b] : 0;
    lo_r = W > 0 ? max(0, P.positions[(long)b * T + tid % T] - W + 1) : 0;
    if (tid % T == 0 && h == 0) {
      if (P.kv_len[b] > ctx_len + T || P.kv_len[b] < 0) set_status(P.status, MLA_DEV_BAD_LENGTH);
      if (W < 0) set_status(P.status, MLA_DEV_BAD_WINDOW);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) lo_r = min(lo_r, __shfl_xor_sync(0xffffffffu, lo_r, o));
  if (lane == 0 && warp < 4) red[warp] = lo_r;
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const int lo_min = min(min(red[0], red[1]), min(red[2], red[3]));
  const int j_lo = lo_min >= ctx_len ? ctx_len / KT * KT : lo_min / KT * KT;
  const int nt_ctx = ctx_len > j_lo ? (ctx_len - j_lo + KT - 1) / KT : 0;
  const int nt = nt_ctx + 1;                                     // + the blocks' own keys
  const uint32_t tmem = B->tmem_slot;
  if (tid == 0) pdl_trigger();

  if (warp == 4 || warp == 6) {
    if (lane == 0) {
      // ---- warp 4: Q, then the key tiles; warp 6: the value tiles ----
      const bool keys = warp == 4;
      if (keys) prefetch_tmap(&P.tmKp);
      prefetch_tmap(&P.tmKV);
      uint64_t* full = keys ? B->kfull : B->vfull;
      uint64_t* empty = keys ? B->kempty : B->vempty;
      bool ok = true;
      for (int t = 0; t < nt && ok; ++t) {
        const int s = t & 1;
        if (!(ok = wait_bar(B, &empty[s], ((t >> 1) & 1) ^ 1, P.status))) break;
        const int row = t < nt_ctx ? coff + j_lo + KT * t : (int)own0;
        uint8_t* slot = keys ? smem + OFF_KR + s * KSLOT : smem + OFF_VR + s * VSLOT;
        mbar_arrive_expect_tx(&full[s], (keys ? 3 : 2) * CH);
        if (t < nt_ctx || !grouped) {
          if (keys) {
            tma_load_3d(slot, &P.tmKV, &full[s], 0, row, 4 * h);            // k_nope (2 chunks)
            tma_load_3d(slot + 2 * CH, &P.tmKp, &full[s], 0, row, 8);       // k_pe
          } else {
            tma_load_3d(slot, &P.tmKV, &full[s], 0, row, 4 * h + 2);        // v (2 chunks)
          }
        } else {
          // the blocks' own keys, block by block (the rest past the end: zeros)
          for (int i = 0; i < slots; ++i) {
            const int r = i < nbu ? P.ctx_rows + unit_block(P, pstart, i) * T : P.rows;
            uint8_t* dst = slot + i * T * 128;
            if (keys) {
              tma_load_3d(dst, &P.tmKVT, &full[s], 0, r, 4 * h);
              tma_load_3d(dst + CH, &P.tmKVT, &full[s], 0, r, 4 * h + 1);
              tma_load_3d(dst + 2 * CH, &P.tmKpT, &full[s], 0, r, 8);
            } else {
              tma_load_3d(dst, &P.tmKVT, &full[s], 0, r, 4 * h + 2);
              tma_load_3d(dst + CH, &P.tmKVT, &full[s], 0, r, 4 * h + 3);
            }
          }
        }
      }
      // every copy into this CTA has landed before it may exit
      if (keys) mbar_wait(&B->q_full, 0, P.status);
      for (int t = max(0, nt - 2); t < nt; ++t) mbar_wait(&full[t & 1], (t >> 1) & 1, P.status);
    }
  } else if (warp == 5 || warp == 7) {
    if (lane == 0) {
      constexpr uint32_t U_CH = CH / 16, U_KSLOT = KSLOT / 16, U_VSLOT = VSLOT / 16, U_KSTEP = 16 * 128 / 16;
      bool ok = true;
      if (warp == 5) {
        // ---- S(t) = [q_nope | q_pe] K(t)^T into S buffer t % NS ----
        const uint32_t id_s16 = idesc_f16(QROWS, KT, true), id_sbf = idesc_f16(QROWS, KT, false);
        const uint64_t dQ = smem_desc_sw128(smem + OFF_Q);
        const uint64_t dK0 = smem_desc_sw128(smem + OFF_KR);
        ok = wait_bar(B, &B->q_full, 0, P.status);
        tc_fence_after();
        for (int t = 0; t < nt && ok; ++t) {
          const int s = t % NS, k = t & 1;
          // S buffer s holds P(t - NS): P(t - NS) V(t - NS) (the other thread)
          // has completed reading it
          if (t >= NS && !(ok = wait_bar(B, &B->o_free[s], (t / NS - 1) & 1, P.status))) break;
          if (!(ok = wait_bar(B, &B->kfull[k], (t >> 1) & 1, P.status))) break;
          tc_fence_after();
          const uint32_t tS = tmem + TM_S + 128 * s;
          const uint64_t dK = dK0 + k * U_KSLOT;
#pragma unroll
          for (int ch = 0; ch < 3; ++ch) {
            const uint32_t id = ch < 2 ? id_s16 : id_sbf;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              mma_f16(tS, dQ + ch * U_CH + 2 * kk, dK + ch * U_CH + 2 * kk, id, (ch | kk) ? 1u : 0u);
          }
          mma_commit(&B->kempty[k]);
          mma_commit(&B->s_full[s]);
        }
      } else {
        // ---- O += P(t) V(t), in tile order ----
        const uint32_t id_pv = idesc_f16_bmn(QROWS, 128, true);
        const uint64_t dV0 = smem_desc_sw128_mn(smem + OFF_VR, CH);
        for (int t = 0; t < nt && ok; ++t) {
          const int s = t % NS, v = t & 1;
          if (!(ok = wait_bar(B, &B->p_full[s], (t / NS) & 1, P.status))) break;
          if (!(ok = wait_bar(B, &B->vfull[v], (t >> 1) & 1, P.status))) break;
          tc_fence_after();
          const uint32_t tP = tmem + TM_S + 128 * s;
          const uint64_t dV = dV0 + v * U_VSLOT;
#pragma unroll
          for (int k = 0; k < KT / 16; ++k)   // 16 keys per MMA: 8 P columns, 16 V rows
            mma_f16_ts(tmem + TM_O, tP + 8 * k, dV + (uint64_t)U_KSTEP * k, id_pv, (t | k) ? 1u : 0u);
          mma_commit(&B->vempty[v]);
          mma_commit(&B->o_free[s]);
        }
      }
      // no MMA of this thread may still run when tensor memory is freed
      uint64_t* drain = warp == 5 ? &B->drain : &B->drain_pv;
      mma_commit(drain);
      mbar_wait(drain, 0, P.status);
    }
  } else if (warp < 4 || warp >= 8) {
    // ---- softmax: row r (TMEM lane r), key columns [64 kh, 64 kh + 64) ----
    const int r = tid & (QROWS - 1), kh = tid >= 256 ? 1 : 0;
    constexpr int KH = KT / 2;
    const uint32_t lane_base = (uint32_t)((r / 32) * 32) << 16;
    const bool live = r < nrows;
    const int bi = r / T, b = unit_block(P, pstart, min(bi, nbu - 1));
    const long m = (long)b * T + (live ? r % T : 0);
    const int p = P.positions[m];
    const bool qv = live && (P.q_visible ? P.q_visible[m] != 0 : true);
    const int W = P.window ? P.window[b] : 0;
    const int kvl = P.kv_len[b];
    // visible keys: context keys [vlo, min(ctx_len, kv_len)); own key i (key
    // ctx_len + i, column bi * T + i of the last tile) for ctx_len + i in
    // [vlo, kv_len), i < T; none for a masked or padding row or a rejected window
    const int vlo = W > 0 ? max(0, p - W + 1) : 0;
    const bool sees = qv && W >= 0;
    const int ctx_hi = sees ? min(ctx_len, kvl) : 0;
    const int own_lo = bi * T + max(0, vlo - ctx_len);
    const int own_hi = sees ? bi * T + min(T, kvl - ctx_len) : 0;
    float mrun = -INFINITY, lsum = 0.f;
    for (int t = 0; t < nt; ++t) {
      const int s = t % NS;
      float sv[KH];
      if (t == max(nt - 3, 0) && live && P.gate) {
        // the epilogue's gate row half, into L2 while the last tiles run
        const float* g = P.gate + m * P.ld_gate + (long)h * 128 + 64 * kh;
        asm volatile("prefetch.global.L2 [%0];" ::"l"(g));
        asm volatile("prefetch.global.L2 [%0];" ::"l"(g + 32));
      }
      wait_bar(B, &B->s_full[s], (t / NS) & 1, P.status);
      tc_fence_after();
#pragma unroll
      for (int q = 0; q < KH; q += 32) tmem_ld32_nowait(tmem + TM_S + 128 * s + KH * kh + q + lane_base, sv + q);
      tmem_ld_wait();
#pragma unroll
      for (int q = 0; q < KH; q += 32) tmem_reg_fence32(sv + q);
      int lo, hi;                                   // visible columns of this tile
      if (t < nt_ctx) {
        const int j0 = j_lo + KT * t;
        lo = max(vlo - j0, 0);
        hi = min(ctx_hi - j0, KT);
      } else {
        lo = own_lo;
        hi = own_hi;
      }
      const int lo_h = lo - KH * kh, hi_h = hi - KH * kh;
      if (!__all_sync(0xffffffffu, lo_h <= 0 && hi_h >= KH)) {
#pragma unroll
        for (int i = 0; i < KH; ++i) sv[i] = (i >= lo_h && i < hi_h) ? sv[i] : -INFINITY;
      }
      float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
      for (int i = 0; i < KH; i += 8) {
#pragma unroll
        for (int j = 0; j < 4; ++j) mx4[j] = max3(mx4[j], sv[i + 2 * j], sv[i + 2 * j + 1]);
      }
      const float hmax = max3(mx4[0], mx4[1], fmaxf(mx4[2], mx4[3]));
      // half maxima exchanged in buffer t % 2: the barrier of tile t + 1
      // orders this tile's reads before the writes of tile t + 2
      float* xmt = xm + (t & 1) * 2 * QROWS;
      xmt[kh * QROWS + r] = hmax;
      pair_sync(warp);
      const float tmax = fmaxf(hmax, xmt[(1 - kh) * QROWS + r]) * P.scale_log2;
      const bool grow = tmax > mrun + RESCALE_LOG2;
      const float m_new = grow ? tmax : mrun;
      const float mref = m_new == -INFINITY ? 0.f : m_new;
      float ps4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int i = 0; i < KH; i += 4) {
        fms2(sv[i], sv[i + 1], P.scale_log2, -mref);
        fms2(sv[i + 2], sv[i + 3], P.scale_log2, -mref);
#pragma unroll
        for (int j = 0; j < 4; ++j) sv[i + j] = fast_exp2(sv[i + j]);
        add2(ps4[0], ps4[1], sv[i], sv[i + 1]);
        add2(ps4[2], ps4[3], sv[i + 2], sv[i + 3]);
      }
      const float psum = (ps4[0] + ps4[1]) + (ps4[2] + ps4[3]);
      const float alpha = (grow && mrun != -INFINITY) ? exp2f(mrun - m_new) : 1.f;
      // P(t - 1) V(t - 1) may still run: a row that grew waits for it, then rescales
      if (t > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
        wait_bar(B, &B->o_free[(t - 1) % NS], ((t - 1) / NS) & 1, P.status);
        tc_fence_after();
#pragma unroll 1
        for (int q = 64 * kh; q < 64 * kh + 64; q += 32) {
          float o[32];
          tmem_ld32(tmem + TM_O + lane_base + q, o);
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] *= alpha;
          tmem_st32(tmem + TM_O + lane_base + q, o);
        }
      }
      lsum = lsum * alpha + psum;
      mrun = m_new;
      // P row in fp16 pairs over S (this thread has read its lane): key 2i in
      // the low half of column i
      {
        uint32_t pw[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          __half2 h2 = __floats2half2_rn(sv[2 * i], sv[2 * i + 1]);
          pw[i] = *reinterpret_cast<uint32_t*>(&h2);
        }
        tmem_st32_u(tmem + TM_S + 128 * s + 32 * kh + lane_base, pw);
      }
      tc_fence_before();
      mbar_arrive(&B->p_full[s]);
    }
    // visibility statistics of the row's token (head 0): its keys form one
    // interval, [vlo, kv_len) clamped to the context and its own block_len
    if (P.vis_stats && h == 0 && kh == 0 && live) {
      const int hi = sees ? min(kvl, ctx_len + T) : 0;
      const int n = max(0, hi - vlo);
      P.vis_stats[m * 3 + 0] = n;
      P.vis_stats[m * 3 + 1] = n ? vlo : -1;
      P.vis_stats[m * 3 + 2] = n ? hi - 1 : -1;
    }
    // ---- epilogue: O / l (times the gate) -> o[m, h, 64 kh .. 64 kh + 63] ----
    float* xmt = xm + (nt & 1) * 2 * QROWS;
    xmt[kh * QROWS + r] = lsum;
    pair_sync(warp);
    lsum += xmt[(1 - kh) * QROWS + r];
    wait_bar(B, &B->o_free[(nt - 1) % NS], ((nt - 1) / NS) & 1, P.status);
    tc_fence_after();
    const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
    __half* dst = P.o + (m * P.H + h) * 128 + 64 * kh;
    const float* g = P.gate && live ? P.gate + m * P.ld_gate + (long)h * 128 + 64 * kh : nullptr;
    // the gate's row piece in 16-byte loads (one wavefront per lane and 16
    // bytes, against one per 4 bytes) when its rows are 16-byte aligned
    const bool g16 = (P.ld_gate & 3) == 0 && ((uintptr_t)P.gate & 15) == 0;
#pragma unroll 1
    for (int q = 0; q < 64; q += 32) {
      float gv[32];
      if (g) {
        if (g16) {
#pragma unroll
          for (int i = 0; i < 32; i += 4) {
            const float4 t4 = *reinterpret_cast<const float4*>(g + q + i);
            gv[i] = t4.x; gv[i + 1] = t4.y; gv[i + 2] = t4.z; gv[i + 3] = t4.w;
          }
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) gv[i] = g[q + i];
        }
      }
      float o[32];
      tmem_ld32(tmem + TM_O + lane_base + 64 * kh + q, o);
      if (live) {
#pragma unroll
        for (int i = 0; i < 32; i += 8) {
          float v[8];
#pragma unroll
          for (int u = 0; u < 8; ++u) v[u] = o[i + u] * inv;
          if (g) {
#pragma unroll
            for (int u = 0; u < 8; ++u) v[u] *= gv[i + u];
          }
          __half2 h2[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) h2[u] = __floats2half2_rn(v[2 * u], v[2 * u + 1]);
          *reinterpret_cast<uint4*>(dst + q + i) = *reinterpret_cast<uint4*>(h2);
        }
      }
    }
  }
  pdl_wait();        // (a no-op for the threads that waited already)
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 5) tmem_dealloc(tmem, TMEM_COLS);
}

// Each context's blocks in the order the units take them: full-mask ones
// (window 0) first, then windowed ones, each class in its given order;
// ncls[c] = (full-mask count, windowed count).  One CTA per context.
__global__ void __launch_bounds__(256) expand_units_kernel(const int32_t* __restrict__ window,
                                                           const int32_t* __restrict__ ctx_start,
                                                           int32_t* __restrict__ perm, int32_t* __restrict__ ncls) {
  __shared__ int wsum[8];
  const int c = blockIdx.x, tid = threadIdx.x, lane = tid % 32, warp = tid / 32;
  const int s = ctx_start[c], e = ctx_start[c + 1];
  pdl_wait();                  // perm may still be read by the kernels before
  int n0 = 0;
  for (int base = s; base < e; base += 256) {
    const int b = base + tid;
    n0 += __syncthreads_count(b < e && (window == nullptr || window[b] == 0));
  }
  int run0 = 0, run1 = 0;
  for (int base = s; base < e; base += 256) {
    const int b = base + tid;
    const bool in = b < e;
    const int f = in && (window == nullptr || window[b] == 0) ? 1 : 0;
    int x = f;                                    // inclusive scan of f over the CTA
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) wsum[warp] = x;
    __syncthreads();
    int before = 0, cnt0 = 0;
#pragma unroll
    for (int w = 0; w < 8; ++w) {
      before += w < warp ? wsum[w] : 0;
      cnt0 += wsum[w];
    }
    __syncthreads();
    const int ex0 = before + x - f;               // full-mask blocks before this one in the chunk
    const int ex1 = min(tid, e - base) - ex0;     // windowed blocks before it
    if (in) perm[f ? s + run0 + ex0 : s + n0 + run1 + ex1] = b;
    run0 += cnt0;
    run1 += min(256, e - base) - cnt0;
  }
  if (tid == 0) {
    ncls[2 * c] = n0;
    ncls[2 * c + 1] = max(e - s, 0) - n0;
  }
}

// One warp per gathered row: context c's key j (rows [coff_c, coff_c +
// ctx_len_c), through the table of c's first block), then block b's own key
// ctx_len + i (rows ctx_rows + b * T + i, zero when past kv_len[b]).
__global__ void __launch_bounds__(256) expand_gather_kernel(
    const __nv_bfloat16* __restrict__ cache, long num_slots, const int32_t* __restrict__ block_table,
    int max_pages, int page_size, const int32_t* __restrict__ kv_len, const int32_t* __restrict__ ctx_len,
    const int32_t* __restrict__ ctx_start, int num_ctx, int ctx_rows, int nb, int T,
    __nv_bfloat16* __restrict__ out, uint32_t* status) {
  const long r = (long)blockIdx.x * 8 + threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  if (r >= (long)ctx_rows + (long)nb * T) return;
  pdl_wait();
  int b = -1, j = 0;
  bool zero = false;
  if (r < ctx_rows) {
    int acc = 0;
    for (int c = 0; c < num_ctx; ++c) {
      if (r < acc + ctx_len[c]) {
        b = ctx_start[c];
        j = (int)(r - acc);
        break;
      }
      acc += ctx_len[c];
    }
  } else {
    const long rr = r - ctx_rows;
    b = (int)(rr / T);
    const int i = (int)(rr % T);
    int c = 0;
    while (c + 1 < num_ctx && ctx_start[c + 1] <= b) ++c;
    j = ctx_len[c] + i;
    zero = j >= kv_len[b];
  }
  uint4* dst = reinterpret_cast<uint4*>(out + r * 576);
  long slot = -1;
  if (b >= 0 && !zero && j / page_size < max_pages) {
    const int pg = block_table[(long)b * max_pages + j / page_size];
    const long sl = (long)pg * page_size + j % page_size;
    if (pg >= 0 && sl < num_slots) slot = sl;
  }
  if (slot < 0 && !zero && lane == 0) set_status(status, MLA_DEV_BAD_PAGE);
  const uint4* src = reinterpret_cast<const uint4*>(cache + (slot < 0 ? 0 : slot) * 576);
  for (int i = lane; i < 72; i += 32) dst[i] = slot < 0 ? make_uint4(0, 0, 0, 0) : src[i];
}

}  // namespace

bool expand_applies(const mla_handle* h, int block_len) {
  const Layout& l = h->lay;
  return h->cfg.dtype == MLA_BF16 && l.rkv == 512 && l.dr == 64 && l.dn == 128 && l.dv == 128 &&
         block_len >= 1 && block_len <= QROWS;
}

void expand_gather(cudaStream_t st, const mla_handle* h, const __nv_bfloat16* cache, int num_pages,
                   const mla_attn_desc_t& d, const mla_shared_ctx_t& ctx, __nv_bfloat16* out, bool pdl) {
  const long rows = expand_rows(ctx, d.num_blocks, d.block_len);
  Launch L(dim3((unsigned)((rows + 7) / 8)), dim3(256), 0, st, pdl);
  cudaLaunchKernelEx(&L.cfg, expand_gather_kernel, cache, (long)num_pages * h->cfg.page_size,
                     d.block_table, (int)d.max_pages, (int)h->cfg.page_size, d.kv_len, ctx.ctx_len,
                     ctx.ctx_block_start, (int)ctx.num_ctx, (int)ctx.ctx_rows, (int)d.num_blocks,
                     (int)d.block_len, out, h->status);
}

mla_status_t expanded_attention(cudaStream_t st, const mla_handle* h, const __half* q_nope,
                                const __nv_bfloat16* q_abs, const __half* kv,
                                const __nv_bfloat16* gathered, long rows, const mla_attn_desc_t& d,
                                const mla_shared_ctx_t& ctx, const int32_t* positions,
                                const float* gate, long ld_gate, __half* o, int32_t* unit_ws, bool pdl) {
  const Layout& l = h->lay;
  if (!expand_applies(h, d.block_len))
    return fail(MLA_ERR_UNSUPPORTED, "expanded attention: needs bf16, kv_lora_rank 512, qk_rope 64, "
                                     "qk_nope 128, v_head 128, block_len <= 128");
  if (d.num_blocks <= 0 || ctx.num_ctx <= 0) return MLA_OK;
  const long M = (long)d.num_blocks * d.block_len;
  ExpParams P;
  if (!make_tmap_chunked(&P.tmQn, true, q_nope, M, (long)l.H * 128, (long)l.H * 128, QROWS, 2) ||
      !make_tmap_chunked(&P.tmQp, false, q_abs, M, (long)l.H * l.L, (long)l.H * l.L, QROWS, 1) ||
      !make_tmap_chunked(&P.tmKV, true, kv, rows, (long)l.H * 256, (long)l.H * 256, KT, 2) ||
      !make_tmap_chunked(&P.tmKp, false, gathered, rows, l.L, l.L, KT, 1))
    return fail(MLA_ERR_CUDA, "expanded attention: cuTensorMapEncodeTiled failed");
  // units of one mask class when a block's rows fill whole 8-row groups of the tile
  const int T = d.block_len;
  const bool grouped = T % 8 == 0 && QROWS % T == 0;
  P.perm = nullptr;
  P.ncls = nullptr;
  if (grouped) {
    if (!make_tmap_chunked(&P.tmQnT, true, q_nope, M, (long)l.H * 128, (long)l.H * 128, T, 1) ||
        !make_tmap_chunked(&P.tmQpT, false, q_abs, M, (long)l.H * l.L, (long)l.H * l.L, T, 1) ||
        !make_tmap_chunked(&P.tmKVT, true, kv, rows, (long)l.H * 256, (long)l.H * 256, T, 1) ||
        !make_tmap_chunked(&P.tmKpT, false, gathered, rows, l.L, l.L, T, 1))
      return fail(MLA_ERR_CUDA, "expanded attention: cuTensorMapEncodeTiled failed");
    Launch U(dim3((unsigned)ctx.num_ctx), dim3(256), 0, st, pdl);
    const cudaError_t eu = cudaLaunchKernelEx(&U.cfg, expand_units_kernel, d.window, ctx.ctx_block_start,
                                              unit_ws, unit_ws + d.num_blocks);
    if (eu != cudaSuccess) return cuda_fail(eu, "expanded attention units launch");
    P.perm = unit_ws;
    P.ncls = unit_ws + d.num_blocks;
  } else {
    P.tmQnT = P.tmQn;
    P.tmQpT = P.tmQp;
    P.tmKVT = P.tmKV;
    P.tmKpT = P.tmKp;
  }
  P.rows = (int)rows;
  P.M = (int)M;
  P.positions = positions;
  P.kv_len = d.kv_len;
  P.window = d.window;
  P.q_visible = d.q_visible;
  P.vis_stats = d.vis_stats;
  P.ctx_len = ctx.ctx_len;
  P.ctx_start = ctx.ctx_block_start;
  P.gate = gate;
  P.ld_gate = ld_gate;
  P.o = o;
  P.status = h->status;
  P.num_ctx = ctx.num_ctx;
  P.ctx_rows = ctx.ctx_rows;
  P.T = d.block_len;
  P.H = l.H;
  P.bpu = QROWS / d.block_len;
  P.scale_log2 = h->scale * 1.4426950408889634f;
  static std::once_flag once;
  std::call_once(once, [] {
    cudaFuncSetAttribute(expand_attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
  });
  // units: each context's blocks (of each mask class) in groups of bpu, at
  // most one partial group per context and class
  const long units = (d.num_blocks + P.bpu - 1) / P.bpu + 2L * ctx.num_ctx;
  Launch L(dim3((unsigned)units, (unsigned)l.H), dim3(THREADS), SMEM_BYTES, st, pdl || grouped);
  const cudaError_t e = cudaLaunchKernelEx(&L.cfg, expand_attn_kernel, P);
  if (e != cudaSuccess) return cuda_fail(e, "expanded attention launch");
  return MLA_OK;
}

}  // namespace tc
}  // namespace mla
