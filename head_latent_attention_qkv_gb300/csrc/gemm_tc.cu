// tcgen05 GEMM for the projections of the MLA draft layer:
//   C[z][m][n] = sum_k A[z][m][k] * B[z][n][k]   (x @ W^T, both K-contiguous)
// with bf16 or fp16 operands, fp32 accumulation in tensor memory, and an
// epilogue that optionally multiplies by sigmoid(G) before storing fp32,
// fp16 or bf16.
//
// One CTA computes a 128 x BN tile.  Warps 0 and 3 (one lane each) stream A
// and B through a shared-memory ring with TMA; one stage holds KBS
// consecutive 64-wide K slices of each operand and arrives in a single copy
// per operand (a chunked 4-D view of the matrix: a TMA copy holds its issuing
// thread for about the same time whatever its size, and copies of different
// warps proceed side by side, so each operand has its own issuing warp and
// few large copies keep the tensor pipe fed).  Warp 1
// (one lane) issues tcgen05.mma (M=128, N=BN, K=16) into a TMEM accumulator
// and frees each stage with tcgen05.commit; warp 2 owns the TMEM allocation.
// All eight warps run the epilogue (with one warp per scheduler its store
// loop was latency-bound: a CTA wrote ~4.6 bytes per cycle).
//
// Split-K (small M): the K range is divided among the `splitk` CTAs of a
// cluster along z.  Every CTA writes its fp32 partial tile to its own shared
// memory; CTA j of the cluster then adds the partials of rows
// [128 j / splitk, 128 (j+1) / splitk) from all of them through distributed
// shared memory, always in rank order (deterministic), applies the epilogue
// and stores.  Without split-K the CTA stages its own tile the same way.  Each
// lane stores 16 bytes and a warp covers whole row pieces (256 to 512 bytes),
// so every store instruction is a coalesced write.
#include "gemm_tc.cuh"

#include <mutex>
#include <type_traits>

#include "tc_ptx.cuh"

namespace mla {
namespace tc {
namespace {

constexpr int BM = 128, BK = 64, THREADS = 256;   // 8 warps: all run the epilogue

// k-blocks per stage and stages by tile width: about 192 KB of ring
template <int BN> struct Cfg;
template <> struct Cfg<64> { static constexpr int KBS = 4, STAGES = 2; };
template <> struct Cfg<128> { static constexpr int KBS = 2, STAGES = 3; };
template <> struct Cfg<256> { static constexpr int KBS = 2, STAGES = 2; };
// the persistent form: the same ring in more, smaller stages, so that more of
// it is in flight while the MMAs read one stage (its tiles run long K loops)
template <int BN> struct PCfg;
template <> struct PCfg<64> { static constexpr int KBS = 2, STAGES = 4; };
template <> struct PCfg<128> { static constexpr int KBS = 1, STAGES = 6; };
template <> struct PCfg<256> { static constexpr int KBS = 1, STAGES = 4; };

template <int BN, typename CF = Cfg<BN>>
struct Smem {
  static constexpr int KBS = CF::KBS, STAGES = CF::STAGES;
  static constexpr int A_BYTES = KBS * BM * BK * 2;
  static constexpr int B_BYTES = KBS * BN * BK * 2;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int RING = STAGES * STAGE_BYTES;
  static constexpr int PITCH = BN * 4 + 16;            // fp32 partial tile row (bank-conflict free)
  static constexpr int BYTES = 1024 /*align slack*/ + RING + 256;
  static_assert(BM * PITCH <= RING, "partial tile fits in the ring");
  static_assert(BYTES <= 232448, "shared memory");
};

// 4-D TMA tile load (coordinates innermost first).
__device__ __forceinline__ void tma_load_4d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int x, int y, int z, int w) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5}], [%6];"
      ::"r"(smem_u32(dst)), "l"((uint64_t)map), "r"(x), "r"(y), "r"(z), "r"(w), "r"(smem_u32(bar))
      : "memory");
}

// Loads of the partial tiles after the cluster barrier (volatile: they stay
// after it); the callers issue all of a row's loads before using any, so
// they are in flight together.
__device__ __forceinline__ float4 ld_peer_v4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(addr));
  return v;
}
__device__ __forceinline__ float4 ld_own_v4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(addr));
  return v;
}

// One 16-byte store of VALS = 16 / sizeof(TC) values.
template <typename TC> __device__ __forceinline__ void store16(TC* dst, const float* o);
template <>
__device__ __forceinline__ void store16<float>(float* dst, const float* o) {
  *reinterpret_cast<float4*>(dst) = make_float4(o[0], o[1], o[2], o[3]);
}
template <typename T16>
__device__ __forceinline__ void store16_16(T16* dst, const float* o) {
  T16 h[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) h[i] = from_f32<T16>(o[i]);
  uint4 u;
  memcpy(&u, h, 16);
  *reinterpret_cast<uint4*>(dst) = u;
}
template <>
__device__ __forceinline__ void store16<__half>(__half* dst, const float* o) {
  store16_16(dst, o);
}
template <>
__device__ __forceinline__ void store16<__nv_bfloat16>(__nv_bfloat16* dst, const float* o) {
  store16_16(dst, o);
}
// The same 16 bytes, packed for a shared-memory staging tile.
template <typename TC> __device__ __forceinline__ uint4 pack16(const float* o) {
  if constexpr (std::is_same<TC, float>::value) {
    return make_uint4(__float_as_uint(o[0]), __float_as_uint(o[1]), __float_as_uint(o[2]), __float_as_uint(o[3]));
  } else {
    TC h[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) h[i] = from_f32<TC>(o[i]);
    uint4 u;
    memcpy(&u, h, 16);
    return u;
  }
}
// 3-D TMA tile store from shared memory (coordinates innermost first) in the
// thread's bulk group; the bulk-group waits below order it against the reuse
// of the staging tile and the kernel's end.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, const void* src, int x, int y, int z) {
  asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%1, %2, %3}], [%4];"
               ::"l"((uint64_t)map), "r"(x), "r"(y), "r"(z), "r"(smem_u32(src)) : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// at most one committed store group still reading shared memory
__device__ __forceinline__ void bulk_wait_read1() { asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory"); }
// every committed store group complete
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

template <int BN, typename TC>
__global__ void __launch_bounds__(THREADS, 1)
gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
               int M, int N, int K, TC* __restrict__ C, long ldc, long sC,
               const float* __restrict__ G, long ldg, long sG, bool gate_act, int sig_from,
               uint32_t idesc, int splitk, int group_m, uint32_t* status) {
  using S = Smem<BN>;
  constexpr int KBS = S::KBS, STAGES = S::STAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint64_t* full = (uint64_t*)(smem + S::RING);
  uint64_t* empty = full + STAGES;
  uint64_t* accum = empty + STAGES;
  uint32_t* tmem_slot = (uint32_t*)(accum + 1);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  // Tile order: CTAs are dispatched x-fastest; with group_m > 1 consecutive
  // CTAs walk group_m row tiles before the next column tile, so the CTAs
  // resident at once share a few rows of A and a few columns of B in L2
  // instead of sweeping all of B (larger than L2) for every row tile.
  int tile_n = blockIdx.x, tile_m = blockIdx.y;
  if (group_m > 1) {
    const long lin = (long)blockIdx.y * gridDim.x + blockIdx.x, per_group = (long)group_m * gridDim.x;
    const int first_m = (int)(lin / per_group) * group_m;
    const int gm = min(group_m, (int)gridDim.y - first_m);
    const long r = lin % per_group;
    tile_m = first_m + (int)(r % gm);
    tile_n = (int)(r / gm);
  }
  const int n0 = tile_n * BN, m0 = tile_m * BM;
  const int z = blockIdx.z / splitk, ks = blockIdx.z % splitk;     // ks == cluster rank
  const int nk = (K + BK - 1) / BK;
  const int ng_all = (nk + KBS - 1) / KBS;                          // stages of the whole K
  const int g0 = (int)((long)ks * ng_all / splitk);                 // this split's stages
  const int ng = (int)((long)(ks + 1) * ng_all / splitk) - g0;
  constexpr uint32_t TMEM_COLS = BN <= 32 ? 32 : BN <= 64 ? 64 : BN <= 128 ? 128 : 256;

  // B (weights) does not depend on the previous kernel: its first stages are
  // requested before anything else, then A once that kernel has finished
  const int first = ng < STAGES ? ng : STAGES;
  if (threadIdx.x == 0) {
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 2);             // one arrival per operand's producer
      mbar_init(&empty[s], 1);
    }
    mbar_init(accum, 1);
    fence_mbar_init();
    for (int g = 0; g < first; ++g) {
      mbar_arrive_expect_tx(&full[g], S::B_BYTES);
      tma_load_4d(smem + g * S::STAGE_BYTES + S::A_BYTES, &tmB, &full[g], 0, n0, (g0 + g) * KBS, z);
    }
    pdl_trigger();
  }
  if (warp == 2) tmem_alloc(tmem_slot, TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_wait();                     // A, the gate and C belong to the kernels around this one

  if ((warp == 0 || warp == 3) && lane == 0) {
    // producers, one copy per stage (KBS k-blocks) each: warp 0 the A
    // operand, warp 3 the B operand past the stages requested above
    const bool is_a = warp == 0;
    bool ok = true;
    for (int g = is_a ? 0 : first; g < ng && ok; ++g) {
      const int s = g % STAGES;
      if (g >= first) ok = mbar_wait(&empty[s], ((g / STAGES) & 1) ^ 1, status);
      if (!ok) break;
      uint8_t* a = smem + s * S::STAGE_BYTES;
      if (is_a) {
        mbar_arrive_expect_tx(&full[s], S::A_BYTES);
        tma_load_4d(a, &tmA, &full[s], 0, m0, (g0 + g) * KBS, z);
      } else {
        mbar_arrive_expect_tx(&full[s], S::B_BYTES);
        tma_load_4d(a + S::A_BYTES, &tmB, &full[s], 0, n0, (g0 + g) * KBS, z);
      }
    }
    // drain: the last loads of every slot have landed before the CTA can exit
    for (int g = max(0, ng - STAGES); g < ng; ++g)
      mbar_wait(&full[g % STAGES], (g / STAGES) & 1, status);
  } else if (warp == 1 && lane == 0) {
    // MMA issuer (k-blocks past K were filled with zeros by TMA and are skipped)
    for (int g = 0; g < ng; ++g) {
      const int s = g % STAGES;
      if (!mbar_wait(&full[s], (g / STAGES) & 1, status)) break;
      tc_fence_after();
      const uint8_t* a = smem + s * S::STAGE_BYTES;
      const uint8_t* b = a + S::A_BYTES;
#pragma unroll
      for (int i = 0; i < KBS; ++i) {
        if ((g0 + g) * KBS + i >= nk) break;
        const uint64_t da = smem_desc_sw128(a + i * BM * BK * 2), db = smem_desc_sw128(b + i * BN * BK * 2);
#pragma unroll
        for (int k = 0; k < BK / 16; ++k)  // advance 16 elements = 32 bytes = 2 descriptor units
          mma_f16(tmem, da + 2 * k, db + 2 * k, idesc, (g | i | k) != 0);
      }
      mma_commit(&empty[s]);
    }
    mma_commit(accum);
  }
  __syncwarp();

  // ---- epilogue: accumulator -> fp32 partial tile in shared memory (the
  // ring is free once the accumulator is complete) ----
  const bool have = ng > 0 && mbar_wait(accum, 0, status);
  tc_fence_after();
  {
    // warp w reads TMEM lanes 32 (w % 4) .. + 31 (its sub-partition), half
    // w / 4 of the columns
    const int q = warp % 4, r = q * 32 + lane;
    const uint32_t lane_addr = tmem + ((uint32_t)(q * 32) << 16);
    float* prow = (float*)(smem + r * S::PITCH);
#pragma unroll 1
    for (int c = (warp / 4) * (BN / 2); c < (warp / 4 + 1) * (BN / 2); c += 32) {
      float v[32];
      if (have) {
        tmem_ld32(lane_addr + c, v);
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = 0.f;
      }
#pragma unroll
      for (int i = 0; i < 32; i += 4)
        *reinterpret_cast<float4*>(prow + c + i) = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (splitk > 1) cluster_sync_all();      // every partial of the cluster is in place
  // ---- sum the partials of this CTA's rows (rank order), epilogue, store:
  // work items are (row, 128-column group); lane l holds columns 4l .. 4l+3
  // of its item; a warp takes items warp, warp + 4, ... four at a time so
  // that their shared-memory loads are in flight together ----
  // work items: VALS consecutive outputs per lane (one 16-byte store), LPR
  // lanes per output row; an item is one warp-wide store of RPI rows (or of
  // one of the CG 32-lane column groups of a row)
  constexpr int VALS = 16 / (int)sizeof(TC), H4 = VALS / 4;
  constexpr int LPR = BN / VALS;
  constexpr int RPI = LPR >= 32 ? 1 : 32 / LPR, CG = LPR >= 32 ? LPR / 32 : 1;
  constexpr int U = VALS == 4 ? 2 : 1, NW = THREADS / 32, MAXS = 8;
  const int r_lo = ks * BM / splitk, r_hi = (ks + 1) * BM / splitk;
  const int items = ((r_hi - r_lo + RPI - 1) / RPI) * CG;
  const int sub = LPR >= 32 ? 0 : lane / LPR;
  const int lcol = (LPR >= 32 ? lane : lane % LPR) * VALS;
  for (int base = warp; base < items; base += U * NW) {
    float acc[U][VALS];
    uint32_t off[U];
    int rr[U], cc[U];
    bool live[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int it = base + u * NW;
      rr[u] = r_lo + (it / CG) * RPI + sub;
      cc[u] = (it % CG) * 32 * VALS + lcol;
      live[u] = it < items && rr[u] < r_hi;
      off[u] = smem_u32(smem + (live[u] ? rr[u] : r_lo) * S::PITCH + (live[u] ? cc[u] : 0) * 4);
#pragma unroll
      for (int i = 0; i < VALS; ++i) acc[u][i] = 0.f;
    }
    if (splitk > 1) {
      // every peer's partial in flight at once, then added in rank order
      // (the same sum in every run)
      float4 t[MAXS][U][H4];
#pragma unroll
      for (int q = 0; q < MAXS; ++q)
        if (q < splitk) {
#pragma unroll
          for (int u = 0; u < U; ++u)
#pragma unroll
            for (int h = 0; h < H4; ++h) t[q][u][h] = ld_peer_v4(mapa(off[u] + 16 * h, (uint32_t)q));
        }
#pragma unroll
      for (int q = 0; q < MAXS; ++q)
        if (q < splitk) {
#pragma unroll
          for (int u = 0; u < U; ++u)
#pragma unroll
            for (int h = 0; h < H4; ++h) {
              acc[u][4 * h] += t[q][u][h].x; acc[u][4 * h + 1] += t[q][u][h].y;
              acc[u][4 * h + 2] += t[q][u][h].z; acc[u][4 * h + 3] += t[q][u][h].w;
            }
        }
    } else {
#pragma unroll
      for (int u = 0; u < U; ++u)
#pragma unroll
        for (int h = 0; h < H4; ++h) {
          const float4 t = ld_own_v4(off[u] + 16 * h);
          acc[u][4 * h] = t.x; acc[u][4 * h + 1] = t.y; acc[u][4 * h + 2] = t.z; acc[u][4 * h + 3] = t.w;
        }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int row = m0 + rr[u], n = n0 + cc[u];
      if (!live[u] || row >= M || n >= N) continue;
      float* o = acc[u];
      if (G) {
        const float* g = G + z * sG + (long)row * ldg + n;
#pragma unroll
        for (int i = 0; i < VALS; ++i)
          if (n + i < N) o[i] = gate_act ? o[i] * g[i] : o[i] / (1.f + expf(-g[i]));
      }
      if (sig_from >= 0) {
#pragma unroll
        for (int i = 0; i < VALS; ++i)
          if (n + i >= sig_from) o[i] = 1.f / (1.f + expf(-o[i]));
      }
      TC* dst = C + z * sC + (long)row * ldc + n;
      if (n + VALS <= N) {
        store16<TC>(dst, o);
      } else {
        for (int i = 0; i < VALS && n + i < N; ++i) dst[i] = from_f32<TC>(o[i]);
      }
    }
  }
  if (splitk > 1) cluster_sync_all();      // no CTA leaves while a peer may still read its partial
  __syncthreads();
  if (warp == 2) tmem_dealloc(tmem, TMEM_COLS);
}

// Persistent form for launches without split-K: one CTA per SM walks the
// tiles (tile c, c + grid, ...), the ring runs on across tiles, and the
// accumulator is double-buffered in tensor memory so that the epilogue of
// one tile (warps 4-7, a thread per row) runs under the next tile's loads
// and MMAs.  The epilogue stages 128 bytes of each of a warp's 32 rows at a
// time in shared memory and writes them with one TMA store (whole lines,
// asynchronous), or, where C's layout does not suit TMA (and for the q_b
// split), stores from registers.  Same warp roles otherwise: warp 0 streams
// A, warp 3 B, warp 1 (one lane) issues the MMAs, warp 2 owns tensor memory.
template <int BN>
struct PSmem {
  static constexpr int STG = Smem<BN, PCfg<BN>>::RING + 1024;   // after the ring and the barriers
  static constexpr int STG_TILE = 32 * 128;                 // a warp's 32 rows x 128 bytes
  static constexpr int BYTES = 1024 + STG + 4 * 2 * STG_TILE;
  static_assert(BYTES <= 232448, "shared memory");
};
struct PBars {
  uint64_t acc_full[2];    // tile accumulator complete (phase per use of the buffer)
  uint64_t acc_empty[2];   // its epilogue has read it (128 arrivals)
  uint64_t drain;          // every MMA of the CTA complete
  uint32_t tmem_slot;
  int abort;
};

__device__ __forceinline__ bool pwait(PBars* B, uint64_t* bar, uint32_t parity, uint32_t* st) {
  if (*(volatile int*)&B->abort) return false;
  if (mbar_wait(bar, parity, st)) return true;
  B->abort = 1;
  return false;
}

template <int BN, typename TC>
__global__ void __launch_bounds__(THREADS, 1)
gemm_tc_persistent(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmR,
                   bool tma_store,
                   int M, int N, int K, TC* __restrict__ C, long ldc, long sC,
                   const float* __restrict__ G, long ldg, long sG, bool gate_act, int sig_from,
                   uint32_t idesc, int group_m, int tiles_n, int tiles_m, int batch, QSplit qs,
                   uint32_t* status) {
  using S = Smem<BN, PCfg<BN>>;
  constexpr int KBS = S::KBS, STAGES = S::STAGES;
  constexpr uint32_t ACC_COLS = BN <= 32 ? 32 : BN <= 64 ? 64 : BN <= 128 ? 128 : 256;
  constexpr uint32_t TMEM_COLS = 2 * ACC_COLS;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint64_t* full = (uint64_t*)(smem + S::RING);
  uint64_t* empty = full + STAGES;
  PBars* PB = (PBars*)(empty + STAGES);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int nk = (K + BK - 1) / BK;
  const int ng = (nk + KBS - 1) / KBS;                              // stages per tile
  const long per_batch = (long)tiles_n * tiles_m, total = per_batch * batch;
  // tile t -> (batch entry, row tile, column tile); row tiles in groups of
  // group_m when that keeps B's columns shared in L2
  auto tile_of = [&](long t, int& z, int& m0, int& n0) {
    z = (int)(t / per_batch);
    const long t_in = t % per_batch;
    int tm, tn;
    if (group_m > 1) {
      const long per_group = (long)group_m * tiles_n;
      const int first_m = (int)(t_in / per_group) * group_m;
      const int gm = min(group_m, tiles_m - first_m);
      const long r = t_in % per_group;
      tm = first_m + (int)(r % gm);
      tn = (int)(r / gm);
    } else {
      tn = (int)(t_in % tiles_n);
      tm = (int)(t_in / tiles_n);
    }
    m0 = tm * BM;
    n0 = tn * BN;
  };

  if (threadIdx.x == 0) {
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 2);             // one arrival per operand's producer
      mbar_init(&empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&PB->acc_full[i], 1);
      mbar_init(&PB->acc_empty[i], 128);
    }
    mbar_init(&PB->drain, 1);
    PB->abort = 0;
    fence_mbar_init();
    pdl_trigger();
  }
  if (warp == 2) tmem_alloc(&PB->tmem_slot, TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = PB->tmem_slot;

  if ((warp == 0 || warp == 3) && lane == 0) {
    // producers: warp 0 the A operand (after the previous kernel), warp 3 the
    // weights (independent of it); one copy per stage each
    const bool is_a = warp == 0;
    if (is_a) pdl_wait();
    long gs = 0;
    bool ok = true;
    for (long t = blockIdx.x; t < total && ok; t += gridDim.x) {
      int z, m0, n0;
      tile_of(t, z, m0, n0);
      for (int g = 0; g < ng && ok; ++g, ++gs) {
        const int s = (int)(gs % STAGES);
        if (!(ok = pwait(PB, &empty[s], (uint32_t)((gs / STAGES) & 1) ^ 1, status))) break;
        uint8_t* a = smem + s * S::STAGE_BYTES;
        if (is_a) {
          mbar_arrive_expect_tx(&full[s], S::A_BYTES);
          tma_load_4d(a, &tmA, &full[s], 0, m0, g * KBS, z);
        } else {
          mbar_arrive_expect_tx(&full[s], S::B_BYTES);
          tma_load_4d(a + S::A_BYTES, &tmB, &full[s], 0, n0, g * KBS, z);
        }
      }
    }
    // drain: the last loads of every slot have landed before the CTA can exit
    for (long g = gs - STAGES < 0 ? 0 : gs - STAGES; g < gs; ++g)
      mbar_wait(&full[g % STAGES], (uint32_t)((g / STAGES) & 1), status);
  } else if (warp == 1 && lane == 0) {
    // MMA issuer (k-blocks past K were filled with zeros by TMA and are skipped)
    long gs = 0;
    int j = 0;
    bool ok = true;
    for (long t = blockIdx.x; t < total && ok; t += gridDim.x, ++j) {
      const int buf = j & 1;
      if (!(ok = pwait(PB, &PB->acc_empty[buf], (uint32_t)((j >> 1) & 1) ^ 1, status))) break;
      tc_fence_after();
      const uint32_t d = tmem + buf * ACC_COLS;
      for (int g = 0; g < ng; ++g, ++gs) {
        const int s = (int)(gs % STAGES);
        if (!(ok = pwait(PB, &full[s], (uint32_t)((gs / STAGES) & 1), status))) break;
        tc_fence_after();
        const uint8_t* a = smem + s * S::STAGE_BYTES;
        const uint8_t* b = a + S::A_BYTES;
#pragma unroll
        for (int i = 0; i < KBS; ++i) {
          if (g * KBS + i >= nk) break;
          const uint64_t da = smem_desc_sw128(a + i * BM * BK * 2), db = smem_desc_sw128(b + i * BN * BK * 2);
#pragma unroll
          for (int k = 0; k < BK / 16; ++k)
            mma_f16(d, da + 2 * k, db + 2 * k, idesc, (g | i | k) != 0);
        }
        mma_commit(&empty[s]);
      }
      if (!ok) break;
      mma_commit(&PB->acc_full[buf]);
    }
    mma_commit(&PB->drain);
    mbar_wait(&PB->drain, 0, status);
  } else if (warp >= 4) {
    // epilogue: thread = accumulator row (TMEM lane 32 (warp % 4) + lane)
    pdl_wait();                        // C and the gate belong to the kernels around this one
    const int q = warp % 4, r = q * 32 + lane;
    const uint32_t lane_addr = (uint32_t)(q * 32) << 16;
    // the gate (W_UV) or the sigmoid of the gate columns (A projection) on
    // 32 values of row `row` from column n
    auto epi_math = [&](float* v, int z, int row, int n) {
      if (G) {
        // the row's 32 gate values (16-byte loads when the row piece is whole and aligned)
        const float* g = G + z * sG + (long)row * ldg + n;
        float gv[32];
        if (n + 32 <= N && ((uintptr_t)g & 15) == 0) {
#pragma unroll
          for (int i = 0; i < 32; i += 4) {
            const float4 t4 = *reinterpret_cast<const float4*>(g + i);
            gv[i] = t4.x; gv[i + 1] = t4.y; gv[i + 2] = t4.z; gv[i + 3] = t4.w;
          }
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) gv[i] = n + i < N ? g[i] : 0.f;
        }
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = gate_act ? v[i] * gv[i] : v[i] / (1.f + expf(-gv[i]));
      }
      if (sig_from >= 0) {
#pragma unroll
        for (int i = 0; i < 32; ++i)
          if (n + i >= sig_from) v[i] = 1.f / (1.f + expf(-v[i]));
      }
    };
    uint8_t* stg_warp = smem + PSmem<BN>::STG + q * 2 * PSmem<BN>::STG_TILE;
    int sbuf = 0;
    int j = 0;
    for (long t = blockIdx.x; t < total; t += gridDim.x, ++j) {
      const int buf = j & 1;
      int z, m0, n0;
      tile_of(t, z, m0, n0);
      const bool ok = pwait(PB, &PB->acc_full[buf], (uint32_t)((j >> 1) & 1), status);
      tc_fence_after();
      const int row = m0 + r;
      if (qs.q_nope) {
        // q_b: 32-column chunks lie inside one head's no-position or RoPE dims
        const int dqk = qs.dn + qs.dr, half = qs.dr / 2;
        int p = 0;
        bool bad = false;
        if (ok && row < M) {
          p = qs.positions[row];
          bad = p < 0 || p >= qs.max_pos;
          if (bad && n0 == 0) set_status(status, MLA_DEV_BAD_POSITION);
        }
        if (tma_store) {
          // staged (dn a multiple of 64, dr 64): a 64-column group is half of
          // one head's no-position dims or all of its RoPE dims, so it leaves
          // as one 128-byte piece per row (fp16 to q_nope through tmC, bf16 to
          // Q_abs's tail through tmR) by the warp's staging tile and one TMA
          // store; rows past M are clipped by the store
#pragma unroll 1
          for (int c0 = 0; c0 < BN; c0 += 64) {
            const int n = n0 + c0, hh = n / dqk, d = n % dqk;
            float v[64];
            tmem_ld32(tmem + buf * ACC_COLS + lane_addr + c0, v);
            tmem_ld32(tmem + buf * ACC_COLS + lane_addr + c0 + 32, v + 32);
            if (n >= N) continue;                       // the same for the whole warp
            const bool rope_dims = d >= qs.dn;
            if (rope_dims) {
              if (qs.interleaved) {
#pragma unroll
                for (int k = 0; k < 32; ++k) {          // pairs (2k, 2k + 1)
                  const float2 cs = bad ? make_float2(0.f, 0.f) : qs.rope[(long)p * half + k];
                  const float a = v[2 * k], bb = v[2 * k + 1];
                  v[2 * k] = a * cs.x - bb * cs.y;
                  v[2 * k + 1] = bb * cs.x + a * cs.y;
                }
              } else {
#pragma unroll
                for (int k = 0; k < 32; ++k) {          // pairs (k, k + 32)
                  const float2 cs = bad ? make_float2(0.f, 0.f) : qs.rope[(long)p * half + k];
                  const float a = v[k], bb = v[k + 32];
                  v[k] = a * cs.x - bb * cs.y;
                  v[k + 32] = bb * cs.x + a * cs.y;
                }
              }
            }
            uint8_t* stg = stg_warp + sbuf * PSmem<BN>::STG_TILE;
            if (lane == 0) bulk_wait_read1();     // the store that last read this tile is done with it
            __syncwarp();
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              const uint4 pk = rope_dims ? pack16<__nv_bfloat16>(v + 8 * k) : pack16<__half>(v + 8 * k);
              *reinterpret_cast<uint4*>(stg + lane * 128 + ((k ^ (lane & 7)) << 4)) = pk;
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0 && ok) {
              if (rope_dims)
                tma_store_3d(&tmR, stg, 0, m0 + 32 * q, hh * (qs.L / 64) + qs.rkv / 64);
              else
                tma_store_3d(&tmC, stg, 0, m0 + 32 * q, hh * (qs.dn / 64) + d / 64);
              bulk_commit();
            }
            sbuf ^= 1;
          }
          tc_fence_before();
          mbar_arrive(&PB->acc_empty[buf]);
          continue;
        }
#pragma unroll 1
        for (int c = 0; c < BN; c += 32) {
          const int n = n0 + c, hh = n / dqk, d = n % dqk;
          float v[32];
          tmem_ld32(tmem + buf * ACC_COLS + lane_addr + c, v);
          const bool second_neox = !qs.interleaved && d >= qs.dn + half;   // done with its partner
          float u[32];
          if (d >= qs.dn && !qs.interleaved && !second_neox)
            tmem_ld32(tmem + buf * ACC_COLS + lane_addr + c + half, u);
          if (!ok || row >= M || n >= N || second_neox) continue;
          const long base = (long)row * qs.H + hh;
          if (d < qs.dn) {
            store16_16(qs.q_nope + base * qs.dn + d, v);
            store16_16(qs.q_nope + base * qs.dn + d + 8, v + 8);
            store16_16(qs.q_nope + base * qs.dn + d + 16, v + 16);
            store16_16(qs.q_nope + base * qs.dn + d + 24, v + 24);
            continue;
          }
          const int rd = d - qs.dn;                       // first RoPE dim of the chunk
          __nv_bfloat16* dst = qs.q_abs + base * qs.L + qs.rkv + rd;
          if (qs.interleaved) {
            // pairs (2k, 2k + 1), k = rd / 2 + i
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const float2 cs = bad ? make_float2(0.f, 0.f) : qs.rope[(long)p * half + rd / 2 + i];
              const float a = v[2 * i], bb = v[2 * i + 1];
              v[2 * i] = a * cs.x - bb * cs.y;
              v[2 * i + 1] = bb * cs.x + a * cs.y;
            }
            store16_16(dst, v); store16_16(dst + 8, v + 8); store16_16(dst + 16, v + 16); store16_16(dst + 24, v + 24);
          } else {
            // pairs (k, k + dr / 2): this chunk holds the first halves, u the second
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const float2 cs = bad ? make_float2(0.f, 0.f) : qs.rope[(long)p * half + rd + i];
              const float a = v[i], bb = u[i];
              v[i] = a * cs.x - bb * cs.y;
              u[i] = bb * cs.x + a * cs.y;
            }
            store16_16(dst, v); store16_16(dst + 8, v + 8); store16_16(dst + 16, v + 16); store16_16(dst + 24, v + 24);
            store16_16(dst + half, u); store16_16(dst + half + 8, u + 8);
            store16_16(dst + half + 16, u + 16); store16_16(dst + half + 24, u + 24);
          }
        }
        tc_fence_before();
        mbar_arrive(&PB->acc_empty[buf]);
        continue;
      }
      if (tma_store) {
        // staged: 128 bytes of each of the warp's rows per chunk into a
        // double-buffered 4 KB tile (128-byte swizzle: 16-byte piece p of row
        // l at p ^ (l % 8), conflict-free stores), written by one TMA store;
        // rows and columns past M and N are clipped by the store
        constexpr int CW = 128 / (int)sizeof(TC), VALS = 16 / (int)sizeof(TC);
        const bool in = ok && row < M;
#pragma unroll 1
        for (int c0 = 0; c0 < BN; c0 += CW) {
          uint8_t* stg = stg_warp + sbuf * PSmem<BN>::STG_TILE;
          if (lane == 0) bulk_wait_read1();     // the store that last read this tile is done with it
          __syncwarp();
#pragma unroll
          for (int h = 0; h < CW; h += 32) {
            float v[32];
            tmem_ld32(tmem + buf * ACC_COLS + lane_addr + c0 + h, v);
            if (in && n0 + c0 + h < N) epi_math(v, z, row, n0 + c0 + h);
#pragma unroll
            for (int k = 0; k < 32 / VALS; ++k) {
              const int piece = h * (int)sizeof(TC) / 16 + k;
              *reinterpret_cast<uint4*>(stg + lane * 128 + ((piece ^ (lane & 7)) << 4)) = pack16<TC>(v + k * VALS);
            }
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0 && ok) {
            tma_store_3d(&tmC, stg, n0 + c0, m0 + 32 * q, z);
            bulk_commit();
          }
          sbuf ^= 1;
        }
        tc_fence_before();
        mbar_arrive(&PB->acc_empty[buf]);
        continue;
      }
#pragma unroll 1
      for (int c = 0; c < BN; c += 32) {
        float v[32];
        tmem_ld32(tmem + buf * ACC_COLS + lane_addr + c, v);
        const int n = n0 + c;
        if (!ok || row >= M || n >= N) continue;
        epi_math(v, z, row, n);
        TC* dst = C + z * sC + (long)row * ldc + n;
        constexpr int VALS = 16 / (int)sizeof(TC);
        if (n + 32 <= N) {
#pragma unroll
          for (int i = 0; i < 32; i += VALS) store16<TC>(dst + i, v + i);
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i)
            if (n + i < N) dst[i] = from_f32<TC>(v[i]);
        }
      }
      tc_fence_before();
      mbar_arrive(&PB->acc_empty[buf]);
    }
    if (tma_store && lane == 0) bulk_wait_all();   // the stores are complete before the CTA ends
    __syncwarp();
  }
  pdl_wait();
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 2) tmem_dealloc(tmem, TMEM_COLS);
}

}  // namespace
}  // namespace tc
}  // namespace mla

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
namespace mla {
namespace tc {
namespace {

using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                              const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                              const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                              CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeFn encode_fn() {
  static EncodeFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = (EncodeFn)p;
  });
  return fn;
}

bool encode(CUtensorMap* m, bool fp16, const void* base, int rank, const cuuint64_t* dims,
            const cuuint64_t* strides, const cuuint32_t* box) {
  EncodeFn enc = encode_fn();
  if (!enc) return false;
  cuuint32_t es[4] = {1, 1, 1, 1};
  return enc(m, fp16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
             (cuuint32_t)rank, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// [batch][rows][K] 16-bit matrix (K contiguous, row stride ld, batch stride
// sbatch elements) viewed as {64, rows, K/64, batch}: a box {64, box_rows,
// kbs, 1} is kbs consecutive 64-wide K slices of box_rows rows.
bool make_operand_map(CUtensorMap* m, bool fp16, const void* base, long rows, long K, long ld,
                      long sbatch, int batch, int box_rows, int kbs) {
  cuuint64_t dims[4] = {64, (cuuint64_t)rows, (cuuint64_t)(K / 64), (cuuint64_t)batch};
  cuuint64_t strides[3] = {(cuuint64_t)ld * 2, 128,
                           (cuuint64_t)(batch > 1 ? sbatch : ld * rows) * 2};
  cuuint32_t box[4] = {64, (cuuint32_t)box_rows, (cuuint32_t)kbs, 1};
  return encode(m, fp16, base, 4, dims, strides, box);
}

// C [batch][M][N] of TC (row stride ldc, batch stride sC elements) as a
// 3-D store map {N, M, batch}, box 128 bytes x 32 rows, 128-byte swizzle;
// false when C's base or strides are not 16-byte multiples (TMA's rule).
template <typename TC>
bool make_store_map(CUtensorMap* m, const void* C, long M, long N, long ldc, long sC, int batch) {
  constexpr long es = sizeof(TC);
  if ((uintptr_t)C % 16 || (ldc * es) % 16 || (batch > 1 && (sC * es) % 16)) return false;
  EncodeFn enc = encode_fn();
  if (!enc) return false;
  const CUtensorMapDataType dt = std::is_same<TC, float>::value ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                 : std::is_same<TC, __half>::value ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                                   : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  cuuint64_t dims[3] = {(cuuint64_t)N, (cuuint64_t)M, (cuuint64_t)batch};
  cuuint64_t strides[2] = {(cuuint64_t)(ldc * es), (cuuint64_t)((batch > 1 ? sC : ldc * M) * es)};
  cuuint32_t box[3] = {(cuuint32_t)(128 / es), 32, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, dt, 3, const_cast<void*>(C), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int num_sms_current();

template <int BN, typename TC>
mla_status_t launch(cudaStream_t st, const GemmArgs& a, int splitk, uint32_t* status) {
  using S = Smem<BN>;
  CUtensorMap ta, tb;
  if (!make_operand_map(&ta, a.fp16, a.A, a.M, a.K, a.lda, a.sA, a.batch, BM, S::KBS) ||
      !make_operand_map(&tb, a.fp16, a.B, a.N, a.K, a.ldb, a.sB, a.batch, BN, S::KBS))
    return fail(MLA_ERR_CUDA, "tcgen05 gemm: cuTensorMapEncodeTiled failed");
  auto kern = gemm_tc_kernel<BN, TC>;
  static std::once_flag once;
  std::call_once(once, [&] {
    cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, S::BYTES);
  });
  Launch L(dim3((a.N + BN - 1) / BN, (a.M + BM - 1) / BM, a.batch * splitk), dim3(THREADS), S::BYTES,
           st, a.pdl, dim3(1, 1, splitk));
  // B of one batch entry larger than a third of L2: walk row tiles in groups
  // of 8 (measured on the DeepSeek-V3-shaped step: 113.3 -> 111.0 ms)
  const double b_bytes = (double)a.N * a.K * 2;
  const int group_m = (b_bytes > 48e6 && (a.M + BM - 1) / BM > 8) ? 8 : 1;
  const int tiles_n = (a.N + BN - 1) / BN, tiles_m = (a.M + BM - 1) / BM;
  const long tiles = (long)tiles_n * tiles_m * a.batch;
  if (a.qsplit_done) *a.qsplit_done = false;
  if (splitk == 1 && tiles > num_sms_current()) {
    // more tiles than SMs: the persistent form, one CTA per SM
    auto pk = gemm_tc_persistent<BN, TC>;
    static std::once_flag once_p;
    std::call_once(once_p, [&] {
      cudaFuncSetAttribute(pk, cudaFuncAttributeMaxDynamicSharedMemorySize, PSmem<BN>::BYTES);
    });
    CUtensorMap tc{}, tr{}, tpa, tpb;
    bool tma_store;
    if (a.qsplit) {
      // the q_b split: staged stores when every 64-column group is one piece
      // of a head's no-position dims or its 64 RoPE dims
      const QSplit& q = *a.qsplit;
      tma_store = BN % 64 == 0 && q.dn % 64 == 0 && q.dr == 64 && q.rkv % 64 == 0 && q.L % 64 == 0 &&
                  a.batch == 1 && a.N == q.H * (q.dn + q.dr) &&
                  make_tmap_chunked(&tc, true, q.q_nope, a.M, (long)q.H * q.dn, (long)q.H * q.dn, 32, 1) &&
                  make_tmap_chunked(&tr, false, q.q_abs, a.M, (long)q.H * q.L, (long)q.H * q.L, 32, 1);
    } else {
      tma_store = make_store_map<TC>(&tc, a.C, a.M, a.N, a.ldc, a.sC, a.batch);
    }
    constexpr int PK = Smem<BN, PCfg<BN>>::KBS;
    if (!make_operand_map(&tpa, a.fp16, a.A, a.M, a.K, a.lda, a.sA, a.batch, BM, PK) ||
        !make_operand_map(&tpb, a.fp16, a.B, a.N, a.K, a.ldb, a.sB, a.batch, BN, PK))
      return fail(MLA_ERR_CUDA, "tcgen05 gemm: cuTensorMapEncodeTiled failed");
    Launch P(dim3((unsigned)num_sms_current()), dim3(THREADS), PSmem<BN>::BYTES, st, a.pdl);
    const cudaError_t ep = cudaLaunchKernelEx(&P.cfg, pk, tpa, tpb, tc, tr, tma_store, a.M, a.N, a.K, (TC*)a.C, a.ldc, a.sC,
                                              a.G, a.ldg, a.sG, a.gate_act, a.sig_from,
                                              idesc_f16(BM, BN, a.fp16), group_m, tiles_n, tiles_m,
                                              a.batch, a.qsplit ? *a.qsplit : QSplit{}, status);
    if (ep != cudaSuccess) return cuda_fail(ep, "tcgen05 gemm launch");
    if (a.qsplit && a.qsplit_done) *a.qsplit_done = true;
    return MLA_OK;
  }
  const cudaError_t e = cudaLaunchKernelEx(&L.cfg, kern, ta, tb, a.M, a.N, a.K, (TC*)a.C, a.ldc, a.sC,
                                           a.G, a.ldg, a.sG, a.gate_act, a.sig_from,
                                           idesc_f16(BM, BN, a.fp16), splitk, group_m, status);
  if (e != cudaSuccess) return cuda_fail(e, "tcgen05 gemm launch");
  return MLA_OK;
}

template <typename TC>
mla_status_t launch_bn(cudaStream_t st, const GemmArgs& a, int bn, int splitk, uint32_t* status) {
  switch (bn) {
    case 64: return launch<64, TC>(st, a, splitk, status);
    case 128: return launch<128, TC>(st, a, splitk, status);
    default: return launch<256, TC>(st, a, splitk, status);
  }
}

int num_sms_current() {
  static int num_sms = 0;
  if (!num_sms) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev);
  }
  return num_sms;
}

// Clusters of s CTAs (one per SM) the GPU holds at once: a cluster lives in
// one GPC and the GPCs differ in size, so this is below sms / s.
long max_active_clusters(int s) {
  static long cache[9] = {};
  if (s <= 1) return num_sms_current();
  if (s > 8) return 0;
  if (!cache[s]) {
    auto kern = gemm_tc_kernel<128, float>;
    cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Smem<128>::BYTES);
    Launch L(dim3(1, 1, s), dim3(THREADS), Smem<128>::BYTES, nullptr, false, dim3(1, 1, s));
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &L.cfg) != cudaSuccess || n <= 0) {
      cudaGetLastError();
      n = num_sms_current() / s;
    }
    cache[s] = n;
  }
  return cache[s];
}

}  // namespace

void plan_gemm(int M, int N, int K, int batch, int out_bytes, int* bn_out, int* split_out) {
  const int nk = (K + BK - 1) / BK;
  const int bns[3] = {256, 128, 64};
  double best = 1e30;
  int best_bn = 64, best_s = 1;
  for (int bn : bns) {
    const double mma = bn == 256 ? 170.0 : 108.0;
    const int kbs = bn == 64 ? 4 : 2;
    const long tiles = (long)((N + bn - 1) / bn) * ((M + BM - 1) / BM) * batch;
    for (int s = 1; s <= (batch == 1 ? 8 : 1); ++s) {
      const long fit = max_active_clusters(s);             // a tile is a cluster of s CTAs
      if (s > 1 && tiles > fit) break;
      if (s > 1 && (nk + kbs - 1) / kbs < s) break;      // at least one stage per split
      const long waves = (tiles + fit - 1) / fit;
      // measured per-CTA costs (cycles): MMAs of its K share; launch,
      // prologue and first copies; with split-K the fp32 partial tile read
      // back through DSMEM (~15 B/cycle) and a cluster barrier per peer;
      // the rows it stores (~14 B/cycle, 16-byte lanes)
      const double mainloop = ((nk + s - 1) / s) * 4.0 * mma;
      const double reduce = s > 1 ? BM * bn * 4.0 / 15.0 + 600.0 * s : 0.0;
      const double store = (double)BM / s * bn * out_bytes / 14.0;
      const double per_cta = mainloop + 3000.0 + reduce + store;
      const double t = waves * per_cta;
      if (t < best * 0.98) { best = t; best_bn = bn; best_s = s; }
    }
  }
  *bn_out = best_bn;
  *split_out = best_s;
}

mla_status_t gemm(cudaStream_t st, const GemmArgs& a, uint32_t* status) {
  if (a.M <= 0 || a.N <= 0 || a.batch <= 0) return MLA_OK;
  const bool ok = a.K % 64 == 0 && a.lda % 8 == 0 && a.ldb % 8 == 0 && a.sA % 8 == 0 &&
                  a.sB % 8 == 0 && a.ldc % (a.out == Out::F32 ? 4 : 8) == 0 &&
                  a.sC % (a.out == Out::F32 ? 4 : 8) == 0 &&
                  (uintptr_t)a.A % 16 == 0 && (uintptr_t)a.B % 16 == 0 &&
                  (uintptr_t)a.C % 16 == 0;
  if (!ok) return fail(MLA_ERR_UNSUPPORTED, "tcgen05 gemm: K must be a multiple of 64, leading dims "
                                             "and strides 16-byte multiples, pointers 16-byte aligned");
  int bn = 64, splitk = 1;
  plan_gemm(a.M, a.N, a.K, a.batch, a.out == Out::F32 ? 4 : 2, &bn, &splitk);
  switch (a.out) {
    case Out::F32: return launch_bn<float>(st, a, bn, splitk, status);
    case Out::F16: return launch_bn<__half>(st, a, bn, splitk, status);
    default: return launch_bn<__nv_bfloat16>(st, a, bn, splitk, status);
  }
}

bool make_tmap_2d(CUtensorMap* m, bool fp16, const void* base, long rows, long cols, long ld,
                  int box_rows) {
  cuuint64_t dims[3] = {(cuuint64_t)cols, (cuuint64_t)rows, 1};
  cuuint64_t strides[2] = {(cuuint64_t)ld * 2, (cuuint64_t)ld * rows * 2};
  cuuint32_t box[3] = {64, (cuuint32_t)box_rows, 1};
  return encode(m, fp16, base, 3, dims, strides, box);
}

bool make_tmap_chunked(CUtensorMap* m, bool fp16, const void* base, long rows, long cols, long ld,
                       int box_rows, int box_chunks) {
  if (cols % 64) return false;
  cuuint64_t dims[3] = {64, (cuuint64_t)rows, (cuuint64_t)(cols / 64)};
  cuuint64_t strides[2] = {(cuuint64_t)ld * 2, 128};
  cuuint32_t box[3] = {64, (cuuint32_t)box_rows, (cuuint32_t)box_chunks};
  return encode(m, fp16, base, 3, dims, strides, box);
}

}  // namespace tc
}  // namespace mla
