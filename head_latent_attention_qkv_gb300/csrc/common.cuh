// Shared host/device definitions of the MLA draft-layer library.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <string>

#include "../../include/mla_draft.h"

namespace mla {

// ---- error reporting (host) -------------------------------------------------
void set_error(const std::string& msg);
mla_status_t fail(mla_status_t s, const std::string& msg);
mla_status_t cuda_fail(cudaError_t e, const char* what);

#define MLA_CUDA_TRY(expr)                                  \
  do {                                                      \
    cudaError_t _e = (expr);                                \
    if (_e != cudaSuccess) return ::mla::cuda_fail(_e, #expr); \
  } while (0)

// ---- element conversion (device) ------------------------------------------
__device__ __forceinline__ float to_f32(float v) { return v; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }
__device__ __forceinline__ float to_f32(__half v) { return __half2float(v); }
template <typename T> __device__ __forceinline__ T from_f32(float v);
template <> __device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v) {
  return __float2bfloat16_rn(v);
}
template <> __device__ __forceinline__ __half from_f32<__half>(float v) { return __float2half_rn(v); }

__device__ __forceinline__ void set_status(uint32_t* status, uint32_t bits) {
  if (status) atomicOr(status, bits);
}

// ---- programmatic dependent launch (device) -----------------------------------
// Every kernel of the library calls pdl_wait() before it touches the outputs
// of earlier kernels of the same call and before it exits, so that a kernel
// started early never completes before its predecessor: completion stays
// ordered along the stream.
// Block until the previous kernel of the stream (when this one was launched
// with programmatic stream serialization) has completed and its writes are
// visible; a no-op otherwise.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// Let the next kernel of the stream start launching (its CTAs are scheduled
// once every CTA of this grid has done this or exited).
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ---- derived layout of one layer (host handle) ------------------------------
struct Layout {
  int D, H, rq, rkv, dn, dr, dv, L, dqk;
  int qdim;        // width of the query block of the A projection: rq or H*dqk
  int gdim;        // gate width (H*dv or 0)
  int NA;          // rows of W_A: L + qdim + gdim, ordered [kv | q | gate]
  size_t elt;      // bytes per element of the configured dtype
  // byte offsets inside the arena
  size_t off_WA, off_Wqb, off_gq, off_gkv, off_WUKT, off_WUV, off_Wo, off_WKV, off_rope, off_status, total;
};

bool make_layout(const mla_config_t& c, Layout* out);

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Launch configuration with optional programmatic stream serialization (the
// kernel may start while the previous kernel of the stream finishes; it calls
// griddepcontrol.wait before touching that kernel's outputs) and optional
// thread-block cluster dimensions.
struct Launch {
  cudaLaunchConfig_t cfg;
  cudaLaunchAttribute attr[2];
  Launch(dim3 grid, dim3 block, size_t smem, cudaStream_t st, bool pdl,
         dim3 cluster = dim3(1, 1, 1)) {
    cfg = cudaLaunchConfig_t{};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    int n = 0;
    if (cluster.x * cluster.y * cluster.z > 1) {
      attr[n].id = cudaLaunchAttributeClusterDimension;
      attr[n].val.clusterDim.x = cluster.x;
      attr[n].val.clusterDim.y = cluster.y;
      attr[n].val.clusterDim.z = cluster.z;
      ++n;
    }
    if (pdl) {
      attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
      attr[n].val.programmaticStreamSerializationAllowed = 1;
      ++n;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
  }
};

}  // namespace mla

struct mla_handle {
  mla_config_t cfg;
  mla::Layout lay;
  int device;
  int num_sms;
  char* arena;
  float scale;     // softmax scale
  uint32_t* status;
  const float2* rope;   // [max_position, dr/2] (cos, sin)
  const float* gamma_q;
  const float* gamma_kv;
  const void* WA;
  const void* Wqb;
  const void* WUKT;     // [H, rkv, dn]
  const void* WUV;      // [H, dv, rkv]
  const void* Wo;
  const void* WKV;       // [H * (dn + dv), rkv] in the layer dtype: kv_b_proj (the expanded form)
  unsigned long long launches;  // kernels enqueued through this handle
};
