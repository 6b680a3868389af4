// tcgen05 GEMM for the projections of the MLA draft layer:
//   C[z][m][n] = sum_k A[z][m][k] * B[z][n][k]   (x @ W^T, both K-contiguous)
// with bf16 or fp16 operands, fp32 accumulation in tensor memory, and an
// epilogue that optionally multiplies by sigmoid(G) before storing fp32,
// fp16 or bf16.
//
// One CTA computes a 128 x BN tile.  Warp 0 (one lane) streams 64-wide K
// slices of A and B through a STAGES-deep shared-memory ring with TMA
// (128-byte swizzle); warp 1 (one lane) issues tcgen05.mma (M=128, N=BN,
// K=16) into a TMEM accumulator and releases each ring slot with
// tcgen05.commit; warp 2 owns the TMEM allocation; after the last commit all
// four warps read the accumulator back (warp w owns TMEM lanes / tile rows
// 32w..32w+31) and store.
#include "gemm_tc.cuh"

#include <mutex>
#include <type_traits>

#include "tc_ptx.cuh"

namespace mla {
namespace tc {
namespace {

constexpr int BM = 128, BK = 64, THREADS = 128;

template <int BN, int STAGES>
struct Smem {
  static constexpr int A_BYTES = BM * BK * 2;
  static constexpr int B_BYTES = BN * BK * 2;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int BYTES = 1024 /*align slack*/ + STAGES * STAGE_BYTES + 256;
};

template <typename TC>
__device__ __forceinline__ void store32(TC* dst, const float* v);
template <>
__device__ __forceinline__ void store32<float>(float* dst, const float* v) {
#pragma unroll
  for (int i = 0; i < 32; i += 4)
    *reinterpret_cast<float4*>(dst + i) = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
}
template <typename T16>
__device__ __forceinline__ void store32_16(T16* dst, const float* v) {
#pragma unroll
  for (int i = 0; i < 32; i += 8) {
    uint4 u;
    T16 h[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) h[j] = from_f32<T16>(v[i + j]);
    memcpy(&u, h, 16);
    *reinterpret_cast<uint4*>(dst + i) = u;
  }
}
template <>
__device__ __forceinline__ void store32<__half>(__half* dst, const float* v) { store32_16(dst, v); }
template <>
__device__ __forceinline__ void store32<__nv_bfloat16>(__nv_bfloat16* dst, const float* v) {
  store32_16(dst, v);
}

template <int BN, int STAGES, typename TC>
__global__ void __launch_bounds__(THREADS, 1)
gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
               int M, int N, int K, TC* __restrict__ C, long ldc, long sC,
               const float* __restrict__ G, long ldg, long sG, uint32_t idesc, int splitk,
               uint32_t* status) {
  using S = Smem<BN, STAGES>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint64_t* full = (uint64_t*)(smem + STAGES * S::STAGE_BYTES);
  uint64_t* empty = full + STAGES;
  uint64_t* accum = empty + STAGES;
  uint32_t* tmem_slot = (uint32_t*)(accum + 1);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int n0 = blockIdx.x * BN, m0 = blockIdx.y * BM;
  const int z = blockIdx.z / splitk, ks = blockIdx.z % splitk;
  const int nk_all = (K + BK - 1) / BK;
  const int kb0 = (int)((long)ks * nk_all / splitk);          // this split's K blocks
  const int nk = (int)((long)(ks + 1) * nk_all / splitk) - kb0;
  constexpr uint32_t TMEM_COLS = BN <= 32 ? 32 : BN <= 64 ? 64 : BN <= 128 ? 128 : 256;

  if (threadIdx.x == 0) {
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(accum, 1);
    fence_mbar_init();
  }
  if (warp == 2) tmem_alloc(tmem_slot, TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0 && lane == 0) {
    // producer: TMA ring; tiles are pulled into L2 2*STAGES k-blocks ahead
    auto prefetch = [&](int kb) {
      if (kb < nk) {
        tma_prefetch_3d(&tmA, (kb0 + kb) * BK, m0, z);
        tma_prefetch_3d(&tmB, (kb0 + kb) * BK, n0, z);
      }
    };
    for (int kb = STAGES; kb < 2 * STAGES; ++kb) prefetch(kb);
    bool ok = true;
    for (int kb = 0; kb < nk && ok; ++kb) {
      const int s = kb % STAGES;
      const uint32_t ph = (kb / STAGES) & 1;
      ok = mbar_wait(&empty[s], ph ^ 1, status);
      if (!ok) break;
      uint8_t* a = smem + s * S::STAGE_BYTES;
      uint8_t* b = a + S::A_BYTES;
      mbar_arrive_expect_tx(&full[s], S::STAGE_BYTES);
      tma_load_3d(a, &tmA, &full[s], (kb0 + kb) * BK, m0, z);
      tma_load_3d(b, &tmB, &full[s], (kb0 + kb) * BK, n0, z);
      prefetch(kb + 2 * STAGES);
    }
    // drain: the last loads of every slot have landed before the CTA can exit
    for (int kb = max(0, nk - STAGES); kb < nk; ++kb)
      mbar_wait(&full[kb % STAGES], (kb / STAGES) & 1, status);
  } else if (warp == 1 && lane == 0) {
    // MMA issuer
    for (int kb = 0; kb < nk; ++kb) {
      const int s = kb % STAGES;
      if (!mbar_wait(&full[s], (kb / STAGES) & 1, status)) break;
      tc_fence_after();
      const uint8_t* a = smem + s * S::STAGE_BYTES;
      const uint8_t* b = a + S::A_BYTES;
      const uint64_t da = smem_desc_sw128(a), db = smem_desc_sw128(b);
#pragma unroll
      for (int k = 0; k < BK / 16; ++k)  // advance 16 elements = 32 bytes = 2 descriptor units
        mma_f16(tmem, da + 2 * k, db + 2 * k, idesc, (kb | k) != 0);
      mma_commit(&empty[s]);
    }
    mma_commit(accum);
  }
  __syncwarp();
  // epilogue: every warp reads its 32 accumulator lanes
  const bool have = nk > 0 && mbar_wait(accum, 0, status);
  tc_fence_after();
  const int row = m0 + warp * 32 + lane;
  const uint32_t lane_addr = tmem + ((uint32_t)(warp * 32) << 16);
#pragma unroll 1
  for (int c = 0; c < BN; c += 32) {
    float v[32];
    tmem_ld32(lane_addr + c, v);
    const int n = n0 + c;
    if (!have || row >= M || n >= N) continue;
    if (G) {
      const float* g = G + z * sG + (long)row * ldg + n;
#pragma unroll
      for (int i = 0; i < 32; ++i)
        if (n + i < N) v[i] = v[i] / (1.f + expf(-g[i]));
    }
    TC* dst = C + z * sC + (long)row * ldc + n;
    if constexpr (std::is_same<TC, float>::value) {
      if (splitk > 1) {
#pragma unroll
        for (int i = 0; i < 32; ++i)
          if (n + i < N) atomicAdd(dst + i, v[i]);
        continue;
      }
    }
    if (n + 32 <= N) {
      store32<TC>(dst, v);
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i)
        if (n + i < N) dst[i] = from_f32<TC>(v[i]);
    }
  }
  tc_fence_before();
  __syncthreads();
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

// [batch][rows][K] 16-bit matrix, K contiguous; box = 64 (K) x box_rows.
bool make_map(CUtensorMap* m, bool fp16, const void* base, long rows, long K, long ld,
              long sbatch, int batch, int box_rows) {
  EncodeFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {(cuuint64_t)K, (cuuint64_t)rows, (cuuint64_t)batch};
  cuuint64_t strides[2] = {(cuuint64_t)ld * 2,
                           (cuuint64_t)(batch > 1 ? sbatch : ld * rows) * 2};
  cuuint32_t box[3] = {64, (cuuint32_t)box_rows, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return enc(m, fp16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
             const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int BN, typename TC>
mla_status_t launch(cudaStream_t st, const GemmArgs& a, uint32_t* status) {
  constexpr int STAGES = 4;
  using S = Smem<BN, STAGES>;
  CUtensorMap ta, tb;
  if (!make_map(&ta, a.fp16, a.A, a.M, a.K, a.lda, a.sA, a.batch, BM) ||
      !make_map(&tb, a.fp16, a.B, a.N, a.K, a.ldb, a.sB, a.batch, BN))
    return fail(MLA_ERR_CUDA, "tcgen05 gemm: cuTensorMapEncodeTiled failed");
  auto kern = gemm_tc_kernel<BN, STAGES, TC>;
  static std::once_flag once;
  std::call_once(once, [&] {
    cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, S::BYTES);
  });
  if (a.splitk > 1) {
    const cudaError_t e = cudaMemset2DAsync(a.C, a.ldc * sizeof(float), 0, a.N * sizeof(float),
                                            (size_t)a.M, st);
    if (e != cudaSuccess) return cuda_fail(e, "tcgen05 gemm: zeroing the split-K output");
  }
  dim3 grid((a.N + BN - 1) / BN, (a.M + BM - 1) / BM, a.batch * a.splitk);
  kern<<<grid, THREADS, S::BYTES, st>>>(ta, tb, a.M, a.N, a.K, (TC*)a.C, a.ldc, a.sC, a.G, a.ldg,
                                         a.sG, idesc_f16(BM, BN, a.fp16), a.splitk, status);
  return MLA_OK;
}

template <typename TC>
mla_status_t launch_bn(cudaStream_t st, const GemmArgs& a, uint32_t* status, int bn) {
  switch (bn) {
    case 64: return launch<64, TC>(st, a, status);
    case 128: return launch<128, TC>(st, a, status);
    case 192: return launch<192, TC>(st, a, status);
    default: return launch<256, TC>(st, a, status);
  }
}

// Tile width: among the widths that give at least one tile per SM, the one
// with the least padded work (ties: the wider tile, fewer A re-reads); if none
// fills the GPU, the narrowest.
int pick_bn(int M, int N, int batch, int num_sms) {
  const int mt = (M + BM - 1) / BM;
  const int cands[4] = {256, 192, 128, 64};
  int best = 0;
  long best_pad = 0;
  for (int bn : cands) {
    const long nt = (N + bn - 1) / bn;
    if ((long)mt * nt * batch < num_sms) continue;
    const long pad = nt * bn - N;
    if (!best || pad < best_pad) { best = bn; best_pad = pad; }
  }
  return best ? best : 64;
}

}  // namespace

int auto_splitk(int M, int N, int K, int batch) {
  static int num_sms = 0;
  if (!num_sms) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev);
  }
  const long tiles = (long)((M + BM - 1) / BM) * ((N + 63) / 64) * batch;
  const int kblocks = (K + BK - 1) / BK;
  if (batch != 1 || tiles >= num_sms || kblocks < 16) return 1;
  int s = (int)((num_sms + tiles - 1) / tiles);
  s = s < kblocks / 8 ? s : kblocks / 8;        // keep >= 8 K blocks per split
  return s < 1 ? 1 : s;
}

mla_status_t gemm(cudaStream_t st, const GemmArgs& a, uint32_t* status) {
  if (a.M <= 0 || a.N <= 0 || a.batch <= 0) return MLA_OK;
  const bool ok = a.K % 8 == 0 && a.lda % 8 == 0 && a.ldb % 8 == 0 && a.sA % 8 == 0 &&
                  a.sB % 8 == 0 && a.ldc % 8 == 0 && a.sC % 8 == 0 &&
                  (uintptr_t)a.A % 16 == 0 && (uintptr_t)a.B % 16 == 0 &&
                  (uintptr_t)a.C % 16 == 0;
  if (!ok) return fail(MLA_ERR_UNSUPPORTED, "tcgen05 gemm: K/leading dims must be multiples of 8 "
                                             "and pointers 16-byte aligned");
  if (a.splitk < 1 || (a.splitk > 1 && (a.out != Out::F32 || a.G || a.batch != 1)))
    return fail(MLA_ERR_INVALID_ARG, "tcgen05 gemm: split-K needs an fp32 output, no gate, batch 1");
  static int num_sms = 0;
  if (!num_sms) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev);
  }
  const int bn = pick_bn(a.M, a.N, a.batch, num_sms);
  switch (a.out) {
    case Out::F32: return launch_bn<float>(st, a, status, bn);
    case Out::F16: return launch_bn<__half>(st, a, status, bn);
    default: return launch_bn<__nv_bfloat16>(st, a, status, bn);
  }
}

}  // namespace tc
}  // namespace mla

namespace mla {
namespace tc {
bool make_tmap_2d(CUtensorMap* m, bool fp16, const void* base, long rows, long cols, long ld,
                  int box_rows) {
  return make_map(m, fp16, base, rows, cols, ld, 0, 1, box_rows);
}
}  // namespace tc
}  // namespace mla

namespace mla {
namespace tc {
// Chunked view of a row-major 16-bit matrix [rows, cols] (row stride ld
// elements, cols a multiple of 64): dims {64, rows, cols / 64}, so that one
// box {64, box_rows, box_chunks} lands in shared memory as box_chunks
// consecutive [box_rows x 128 B] blocks, each 128-byte swizzled -- several
// 64-column K-major operand tiles in one TMA copy.
bool make_tmap_chunked(CUtensorMap* m, bool fp16, const void* base, long rows, long cols, long ld,
                       int box_rows, int box_chunks) {
  EncodeFn enc = encode_fn();
  if (!enc || cols % 64) return false;
  cuuint64_t dims[3] = {64, (cuuint64_t)rows, (cuuint64_t)(cols / 64)};
  cuuint64_t strides[2] = {(cuuint64_t)ld * 2, 128};
  cuuint32_t box[3] = {64, (cuuint32_t)box_rows, (cuuint32_t)box_chunks};
  cuuint32_t es[3] = {1, 1, 1};
  return enc(m, fp16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
             const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
}  // namespace tc
}  // namespace mla
