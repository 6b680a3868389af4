// tcgen05 GEMM launcher (see gemm_tc.cu).
#pragma once

#include <cuda.h>

#include "common.cuh"

namespace mla {
namespace tc {

enum class Out { F32, F16, BF16 };

// q_b epilogue: for each head, the no-position dims go to q_nope (fp16)
// and the RoPE dims, rotated by the row's position, to the tail of Q_abs
// (bf16), instead of C.
struct QSplit {
  __half* q_nope;                 // [rows, H, dn]
  __nv_bfloat16* q_abs;           // [rows, H, L]: dims rkv .. rkv + dr written
  const int32_t* positions;       // [rows]
  const float2* rope;             // [max_pos, dr / 2] (cos, sin)
  int H, dn, dr, L, rkv, max_pos, interleaved;
};

struct GemmArgs {
  int M, N, K, batch;
  bool fp16;                 // operand type: fp16 (true) or bf16 (false)
  const void* A; long lda, sA;   // [batch][M][K] (elements; lda, sA strides)
  const void* B; long ldb, sB;   // [batch][N][K]
  void* C; long ldc, sC; Out out;
  const float* G; long ldg, sG;  // optional gate, same indexing as C: C *= sigmoid(G)
  bool pdl = false;              // may start while the previous kernel of the stream finishes
  bool gate_act = false;         // G already holds sigmoid(gate): C *= G
  int sig_from = -1;             // columns n >= sig_from (>= 0) of C store sigmoid(value)
  const QSplit* qsplit = nullptr;  // q_b split/rotation in the epilogue (persistent launches)
  bool* qsplit_done = nullptr;     // set true when the launch did it (C then not written)
};

// Tile width (64, 128 or 256 columns) and split-K factor (CTAs of a cluster
// along K, 1 = none) the launcher uses for this shape.
void plan_gemm(int M, int N, int K, int batch, int out_bytes, int* bn, int* splitk);

// Enqueue C = A B^T (* sigmoid(G), or * G when gate_act; sigmoid applied to
// the columns from sig_from on) on `st`.  When the output tiles alone do
// not fill the GPU (and batch == 1) K is split over a cluster of CTAs whose
// fp32 partials are added in shared memory, in a fixed order, before the
// epilogue: no atomics, no zeroing, any output type.  Returns
// MLA_ERR_UNSUPPORTED for shapes the kernel does not take (K not a multiple
// of 64, leading dims not multiples of 8, unaligned pointers) and
// MLA_ERR_CUDA if the tensor maps cannot be built or the launch fails.
mla_status_t gemm(cudaStream_t st, const GemmArgs& a, uint32_t* status);

}  // namespace tc
}  // namespace mla

namespace mla {
namespace tc {
// Tensor map of a row-major 16-bit matrix [rows, cols] (row stride ld
// elements), box = 64 columns x box_rows rows, 128-byte swizzle.  The map has
// rank 3 (a unit batch dimension): load it with 3-D TMA, z = 0.
bool make_tmap_2d(CUtensorMap* m, bool fp16, const void* base, long rows, long cols, long ld,
                  int box_rows);
// The same matrix viewed as {64, rows, cols / 64}: a box {64, box_rows,
// box_chunks} brings box_chunks 64-column tiles ([box_rows x 128 B] each,
// 128-byte swizzled, consecutive in shared memory) in one copy.  Load it
// with 3-D TMA at coordinates (0, row, first chunk).
bool make_tmap_chunked(CUtensorMap* m, bool fp16, const void* base, long rows, long cols, long ld,
                       int box_rows, int box_chunks);
}  // namespace tc
}  // namespace mla
