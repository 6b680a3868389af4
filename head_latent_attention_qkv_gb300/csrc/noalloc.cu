// Latent-cache append that allocates nothing and needs no caller workspace.
//
// mla_latent_cache_append() stages the raw [n, kv_lora_rank + qk_rope] fp32
// projection in a workspace the caller allocates.  Some callers cannot
// allocate device memory at the point where they append: code running inside
// a host callback or a custom allocator hook, runtimes whose memory pool is
// fixed before the model starts, or embedders that only hand over the tensors
// they already own.  This variant stages the projection in a fixed
// file-scope device array instead, so the caller passes only inputs and
// outputs.
#include <mutex>
#include <unordered_map>

#include "common.cuh"
#include "simt.cuh"

namespace {

// 4 MiB of staging, held by every GPU that loads the library until exit.
constexpr long kScratchFloats = 1L << 20;
static __device__ __align__(256) float g_append_scratch[kScratchFloats];

std::mutex g_mu;
std::unordered_map<int, float*> g_scratch_addr;  // device ordinal -> address of the array

// The array's name is only a host-side stand-in in host code; its device
// address is looked up once per device, with that device current, and kept for
// the life of the process (a device reset would destroy the array; the header
// rules out calls after one).
mla_status_t scratch_for_current_device(float** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return mla::cuda_fail(e, "append_noalloc: cudaGetDevice");
  std::lock_guard<std::mutex> lock(g_mu);
  auto it = g_scratch_addr.find(dev);
  if (it != g_scratch_addr.end()) {
    *out = it->second;
    return MLA_OK;
  }
  float* p = nullptr;
  e = cudaGetSymbolAddress((void**)&p, g_append_scratch);
  if (e != cudaSuccess) return mla::cuda_fail(e, "append_noalloc: cudaGetSymbolAddress");
  g_scratch_addr[dev] = p;
  *out = p;
  return MLA_OK;
}

}  // namespace

extern "C" int64_t mla_append_noalloc_max_tokens(const mla_handle_t* h) {
  return h ? kScratchFloats / h->lay.L : 0;
}

extern "C" mla_status_t mla_latent_cache_append_noalloc(mla_handle_t* h, const void* hidden,
                                                        const int32_t* positions,
                                                        const int64_t* slot_mapping, int32_t n,
                                                        void* cache, int32_t num_pages,
                                                        void* stream) {
  using namespace mla;
  if (!h) return fail(MLA_ERR_INVALID_ARG, "append_noalloc: null handle");
  if (n < 0) return fail(MLA_ERR_INVALID_ARG, "append_noalloc: n < 0");
  if (n == 0) return MLA_OK;
  if (!hidden || !positions || !slot_mapping || !cache)
    return fail(MLA_ERR_INVALID_ARG, "append_noalloc: null pointer");
  if (num_pages <= 0) return fail(MLA_ERR_INVALID_ARG, "append_noalloc: num_pages <= 0");
  const Layout& l = h->lay;
  if ((long)n * l.L > kScratchFloats)
    return fail(MLA_ERR_INVALID_ARG,
                "append_noalloc: n = " + std::to_string(n) + " tokens exceeds the fixed scratch (" +
                    std::to_string(kScratchFloats / l.L) + " tokens at this entry width); "
                    "split the append or use mla_latent_cache_append");
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "append_noalloc: cudaGetDevice");
  if (dev != h->device)
    return fail(MLA_ERR_INVALID_ARG, "append_noalloc: the handle's device is not the current device");
  float* kv = nullptr;
  mla_status_t s = scratch_for_current_device(&kv);
  if (s != MLA_OK) return s;
  cudaStream_t st = (cudaStream_t)stream;
  const long num_slots = (long)num_pages * h->cfg.page_size;
  // Every staged element the finish step reads is written by the projection
  // first, so nothing in the array has to start at zero.
  if (h->cfg.dtype == MLA_BF16) {
    using T = __nv_bfloat16;
    simt::gemm_nt<T, float>(st, n, l.L, l.D, 1, (const T*)hidden, l.D, 0, (const T*)h->WA, l.D, 0,
                            kv, l.L, 0, nullptr, 0, 0);
    simt::kv_finish<T>(st, h, kv, l.L, n, positions, slot_mapping, (T*)cache, num_slots);
  } else {
    simt::gemm_nt<float, float>(st, n, l.L, l.D, 1, (const float*)hidden, l.D, 0,
                                (const float*)h->WA, l.D, 0, kv, l.L, 0, nullptr, 0, 0);
    simt::kv_finish<float>(st, h, kv, l.L, n, positions, slot_mapping, (float*)cache, num_slots);
  }
  h->launches += 2;
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "append_noalloc: launch");
  return MLA_OK;
}
