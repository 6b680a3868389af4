// C ABI of the MLA draft-layer library: validation, derived-weight arena,
// launch sequences (include/mla_draft.h documents every entry point).
#include <math.h>
#include <string.h>

#include <string>
#include <type_traits>
#include <vector>

#include "common.cuh"
#include "append_tc.cuh"
#include "attn_tc.cuh"
#include "decode_tc.cuh"
#include "expand_tc.cuh"
#include "gemm_tc.cuh"
#include "simt.cuh"

namespace mla {

static thread_local std::string g_last_error;

void set_error(const std::string& msg) { g_last_error = msg; }

mla_status_t fail(mla_status_t s, const std::string& msg) {
  g_last_error = msg;
  return s;
}

mla_status_t cuda_fail(cudaError_t e, const char* what) {
  g_last_error = std::string(what) + ": " + cudaGetErrorString(e);
  return MLA_ERR_CUDA;
}

// Arena layout: W_A [NA, D] (rows [kv | q | gate]), W_qb [H*dqk, rq],
// gamma_q fp32 [rq], gamma_kv fp32 [rkv], W_UK^T [H, rkv, dn],
// W_UV [H, dv, rkv], W_o [D, H*dv], kv_b_proj [H*(dn+dv), rkv] (the expanded
// form's K/V expansion, layer dtype), rope float2 [max_pos, dr/2], status.
bool make_layout(const mla_config_t& c, Layout* out) {
  Layout l;
  l.D = c.hidden_size; l.H = c.num_heads; l.rq = c.q_lora_rank; l.rkv = c.kv_lora_rank;
  l.dn = c.qk_nope_head_dim; l.dr = c.qk_rope_head_dim; l.dv = c.v_head_dim;
  if (l.D <= 0 || l.H <= 0 || l.rq < 0 || l.rkv <= 0 || l.dn <= 0 || l.dr <= 0 || l.dv <= 0)
    return false;
  if (l.dr % 2 || c.page_size <= 0 || c.max_position <= 0) return false;
  if (c.dtype != MLA_BF16 && c.dtype != MLA_FP32) return false;
  if (c.rope != MLA_ROPE_NEOX && c.rope != MLA_ROPE_INTERLEAVED) return false;
  l.L = l.rkv + l.dr;
  l.dqk = l.dn + l.dr;
  l.qdim = l.rq > 0 ? l.rq : l.H * l.dqk;
  l.gdim = c.use_output_gate ? l.H * l.dv : 0;
  l.NA = l.L + l.qdim + l.gdim;
  l.elt = c.dtype == MLA_BF16 ? 2 : 4;
  size_t o = 0;
  l.off_WA = o;   o = align256(o + (size_t)l.NA * l.D * l.elt);
  l.off_Wqb = o;  o = align256(o + (l.rq > 0 ? (size_t)l.H * l.dqk * l.rq * l.elt : 0));
  l.off_gq = o;   o = align256(o + (size_t)l.rq * 4);
  l.off_gkv = o;  o = align256(o + (size_t)l.rkv * 4);
  l.off_WUKT = o; o = align256(o + (size_t)l.H * l.rkv * l.dn * l.elt);
  l.off_WUV = o;  o = align256(o + (size_t)l.H * l.dv * l.rkv * l.elt);
  l.off_Wo = o;   o = align256(o + (size_t)l.D * l.H * l.dv * l.elt);
  l.off_WKV = o;  o = align256(o + (size_t)l.H * (l.dn + l.dv) * l.rkv * l.elt);
  l.off_rope = o; o = align256(o + (size_t)c.max_position * (l.dr / 2) * sizeof(float2));
  l.off_status = o; o = align256(o + 256);
  l.total = o;
  *out = l;
  return true;
}

}  // namespace mla

using namespace mla;

extern "C" {

const char* mla_status_string(mla_status_t s) {
  switch (s) {
    case MLA_OK: return "ok";
    case MLA_ERR_INVALID_ARG: return "invalid argument";
    case MLA_ERR_UNSUPPORTED: return "unsupported configuration";
    case MLA_ERR_CUDA: return "CUDA error";
    case MLA_ERR_DEVICE_CHECK: return "device index check failed";
    case MLA_ERR_TIMEOUT: return "device wait timed out";
    default: return "unknown status";
  }
}

const char* mla_last_error(void) { return g_last_error.c_str(); }

int32_t mla_cache_entry_dim(const mla_config_t* cfg) {
  Layout l;
  if (!cfg || !make_layout(*cfg, &l)) return 0;
  return l.L;
}

size_t mla_cache_page_bytes(const mla_config_t* cfg) {
  Layout l;
  if (!cfg || !make_layout(*cfg, &l)) return 0;
  return (size_t)cfg->page_size * 1 /* one latent KV head */ * l.L * l.elt;
}

size_t mla_weight_arena_bytes(const mla_config_t* cfg) {
  Layout l;
  if (!cfg || !make_layout(*cfg, &l)) return 0;
  return l.total;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Init: validation and re-layout of the weights into the arena
// ---------------------------------------------------------------------------
namespace mla {
namespace {

template <typename T>
__global__ void to_f32_kernel(const T* __restrict__ in, float* __restrict__ out, int n) {
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x)
    out[i] = to_f32(in[i]);
}

template <typename TI, typename TO>
__global__ void convert_kernel(const TI* __restrict__ in, TO* __restrict__ out, long n) {
  for (long i = blockIdx.x * (long)blockDim.x + threadIdx.x; i < n; i += (long)gridDim.x * blockDim.x)
    out[i] = from_f32<TO>(to_f32(in[i]));
}

// W_UV[h][v][c] = kv_b_proj[h*(dn+dv) + dn + v][c]   (v < dv, c < rkv)
template <typename TI, typename TO>
__global__ void wuv_gather_kernel(const TI* __restrict__ kvb, TO* __restrict__ out, int H, int dn,
                                  int dv, int rkv) {
  const long total = (long)H * dv * rkv;
  for (long idx = blockIdx.x * (long)blockDim.x + threadIdx.x; idx < total;
       idx += (long)gridDim.x * blockDim.x) {
    const int c = idx % rkv;
    const int v = (idx / rkv) % dv;
    const int h = idx / ((long)rkv * dv);
    out[idx] = from_f32<TO>(to_f32(kvb[((long)h * (dn + dv) + dn + v) * rkv + c]));
  }
}

// W_UK^T[h][c][i] = kv_b_proj[h*(dn+dv) + i][c]   (i < dn, c < rkv)
template <typename TI, typename TO>
__global__ void wuk_transpose_kernel(const TI* __restrict__ kvb, TO* __restrict__ out, int H,
                                     int dn, int dv, int rkv) {
  const long total = (long)H * rkv * dn;
  for (long idx = blockIdx.x * (long)blockDim.x + threadIdx.x; idx < total;
       idx += (long)gridDim.x * blockDim.x) {
    const int i = idx % dn;
    const int c = (idx / dn) % rkv;
    const int h = idx / ((long)dn * rkv);
    out[idx] = from_f32<TO>(to_f32(kvb[((long)h * (dn + dv) + i) * rkv + c]));
  }
}

// Derived weights that meet the intermediate activations (W_qb, W_UK^T, W_UV,
// W_o) are stored in the intermediate type TO (fp16 for bf16 layers, an
// exact conversion for weights of normal magnitude).
template <typename TI, typename TO>
void relayout_weights(const Layout& l, const mla_weights_t& w, char* a, cudaStream_t st) {
  const int G = 1024, B = 256;
  if (l.rq > 0) {
    convert_kernel<TI, TO><<<G, B, 0, st>>>((const TI*)w.q_b_proj, (TO*)(a + l.off_Wqb),
                                            (long)l.H * l.dqk * l.rq);
    convert_kernel<TI, float><<<8, B, 0, st>>>((const TI*)w.q_a_layernorm, (float*)(a + l.off_gq), l.rq);
  }
  convert_kernel<TI, float><<<8, B, 0, st>>>((const TI*)w.kv_a_layernorm, (float*)(a + l.off_gkv), l.rkv);
  wuk_transpose_kernel<TI, TO><<<G, B, 0, st>>>((const TI*)w.kv_b_proj, (TO*)(a + l.off_WUKT), l.H,
                                                 l.dn, l.dv, l.rkv);
  wuv_gather_kernel<TI, TO><<<G, B, 0, st>>>((const TI*)w.kv_b_proj, (TO*)(a + l.off_WUV), l.H,
                                              l.dn, l.dv, l.rkv);
  convert_kernel<TI, TO><<<G, B, 0, st>>>((const TI*)w.o_proj, (TO*)(a + l.off_Wo),
                                          (long)l.D * l.H * l.dv);
  convert_kernel<TI, TI><<<G, B, 0, st>>>((const TI*)w.kv_b_proj, (TI*)(a + l.off_WKV),
                                          (long)l.H * (l.dn + l.dv) * l.rkv);
}

mla_status_t validate(const mla_config_t& c, const mla_weights_t& w, Layout* l) {
  if (!make_layout(c, l))
    return fail(MLA_ERR_INVALID_ARG,
                "config: dims must be positive (q_lora_rank >= 0), qk_rope_head_dim even, "
                "page_size/max_position positive, dtype and rope valid");
  if (!(c.rope_theta > 0) || !(c.rms_norm_eps >= 0) || !(c.softmax_scale >= 0))
    return fail(MLA_ERR_INVALID_ARG, "config: rope_theta > 0, rms_norm_eps >= 0, softmax_scale >= 0");
  if (c.q_lora_rank > 0) {
    if (!w.fused_qkv_a_proj || !w.q_a_layernorm || !w.q_b_proj)
      return fail(MLA_ERR_INVALID_ARG, "weights: q_lora_rank > 0 needs fused_qkv_a_proj, q_a_layernorm, q_b_proj");
  } else if (!w.q_proj || !w.kv_a_proj_with_mqa) {
    return fail(MLA_ERR_INVALID_ARG, "weights: q_lora_rank == 0 needs q_proj and kv_a_proj_with_mqa");
  }
  if (!w.kv_a_layernorm || !w.kv_b_proj || !w.o_proj)
    return fail(MLA_ERR_INVALID_ARG, "weights: kv_a_layernorm, kv_b_proj and o_proj are required");
  if (c.use_output_gate && !w.gate_proj)
    return fail(MLA_ERR_INVALID_ARG, "weights: use_output_gate needs gate_proj");
  if (l->rkv % 16 || l->rkv > 512)
    return fail(MLA_ERR_UNSUPPORTED, "kv_lora_rank must be a multiple of 16 and at most 512");
  if (l->L > 1024)
    return fail(MLA_ERR_UNSUPPORTED, "kv_lora_rank + qk_rope_head_dim must be at most 1024");
  if (c.dtype == MLA_BF16) {
    // the tensor-core kernels: latent attention on 512 + 64 dims, 64-wide K
    // slices in every projection, 16-byte output rows
    const int ps = c.page_size;
    if (l->rkv != 512 || l->dr != 64)
      return fail(MLA_ERR_UNSUPPORTED, "bf16 layers: kv_lora_rank 512 and qk_rope_head_dim 64");
    if (ps % 16 || (ps < 128 && 128 % ps) || (ps > 128 && ps % 128))
      return fail(MLA_ERR_UNSUPPORTED, "bf16 layers: page_size 16, 32, 64 or a multiple of 128");
    if (l->D % 64 || l->rq % 64 || l->dn % 64 || (l->H * l->dv) % 64 || l->dv % 8)
      return fail(MLA_ERR_UNSUPPORTED, "bf16 layers: hidden_size, q_lora_rank, qk_nope_head_dim and "
                                       "num_heads * v_head_dim multiples of 64, v_head_dim of 8");
  }
  return MLA_OK;
}

}  // namespace
}  // namespace mla

extern "C" mla_status_t mla_draft_init(const mla_config_t* cfg, const mla_weights_t* w,
                                       void* arena, size_t arena_bytes, void* stream,
                                       mla_handle_t** out) {
  if (!cfg || !w || !arena || !out) return fail(MLA_ERR_INVALID_ARG, "init: null argument");
  *out = nullptr;
  Layout l;
  mla_status_t s = validate(*cfg, *w, &l);
  if (s != MLA_OK) return s;
  if (arena_bytes < l.total)
    return fail(MLA_ERR_INVALID_ARG, "init: arena smaller than mla_weight_arena_bytes()");
  if ((uintptr_t)arena % 256)
    return fail(MLA_ERR_INVALID_ARG, "init: arena must be 256-byte aligned");
  cudaStream_t st = (cudaStream_t)stream;
  auto* h = new mla_handle();
  h->cfg = *cfg;
  h->lay = l;
  h->arena = (char*)arena;
  {
    cudaError_t e0 = cudaGetDevice(&h->device);
    if (e0 == cudaSuccess)
      e0 = cudaDeviceGetAttribute(&h->num_sms, cudaDevAttrMultiProcessorCount, h->device);
    if (e0 != cudaSuccess) { delete h; return cuda_fail(e0, "init: device query"); }
  }
  h->scale = cfg->softmax_scale > 0 ? (float)cfg->softmax_scale : (float)(1.0 / sqrt((double)l.dqk));
  char* a = h->arena;
  h->WA = a + l.off_WA; h->Wqb = a + l.off_Wqb; h->WUKT = a + l.off_WUKT; h->WUV = a + l.off_WUV;
  h->Wo = a + l.off_Wo; h->WKV = a + l.off_WKV; h->gamma_q = (float*)(a + l.off_gq); h->gamma_kv = (float*)(a + l.off_gkv);
  h->rope = (float2*)(a + l.off_rope); h->status = (uint32_t*)(a + l.off_status);
  const size_t e = l.elt, rowb = (size_t)l.D * e;
  char* WA = a + l.off_WA;
  const char* kv_src = cfg->q_lora_rank > 0 ? (const char*)w->fused_qkv_a_proj + (size_t)l.rq * rowb
                                            : (const char*)w->kv_a_proj_with_mqa;
  const char* q_src = cfg->q_lora_rank > 0 ? (const char*)w->fused_qkv_a_proj : (const char*)w->q_proj;
  cudaError_t err = cudaSuccess;
#define STEP(x) if (err == cudaSuccess) err = (x)
  STEP(cudaMemcpyAsync(WA, kv_src, (size_t)l.L * rowb, cudaMemcpyDeviceToDevice, st));
  STEP(cudaMemcpyAsync(WA + (size_t)l.L * rowb, q_src, (size_t)l.qdim * rowb, cudaMemcpyDeviceToDevice, st));
  if (l.gdim)
    STEP(cudaMemcpyAsync(WA + (size_t)(l.L + l.qdim) * rowb, w->gate_proj, (size_t)l.gdim * rowb,
                         cudaMemcpyDeviceToDevice, st));
  STEP(cudaMemsetAsync(a + l.off_status, 0, 256, st));
  if (err != cudaSuccess) { delete h; return cuda_fail(err, "init: weight copy"); }
  if (cfg->dtype == MLA_BF16)
    relayout_weights<__nv_bfloat16, __half>(l, *w, a, st);
  else
    relayout_weights<float, float>(l, *w, a, st);
  // RoPE table: angle = pos * theta^(-2k/dr), cos/sin evaluated in double.
  const int half = l.dr / 2;
  std::vector<float2> tab((size_t)cfg->max_position * half);
  for (int k = 0; k < half; ++k) {
    const double inv = pow(cfg->rope_theta, -2.0 * k / l.dr);
    for (int p = 0; p < cfg->max_position; ++p) {
      const double ang = (double)p * inv;
      tab[(size_t)p * half + k] = make_float2((float)cos(ang), (float)sin(ang));
    }
  }
  STEP(cudaMemcpyAsync(a + l.off_rope, tab.data(), tab.size() * sizeof(float2),
                       cudaMemcpyHostToDevice, st));
  STEP(cudaGetLastError());
  STEP(cudaStreamSynchronize(st));
#undef STEP
  if (err != cudaSuccess) { delete h; return cuda_fail(err, "init: relayout"); }
  *out = h;
  return MLA_OK;
}

extern "C" void mla_draft_destroy(mla_handle_t* h) { delete h; }

// ---------------------------------------------------------------------------
// Workspace
// ---------------------------------------------------------------------------
namespace mla {
namespace {

struct FwdWs {
  size_t a_out, q_cn, q_raw, q_nope, q_abs, o_lat, o, dec, dec_bytes, total;
};

// Bytes the few-row attention may need for a forward of M block tokens: it
// applies only when block_len * num_heads <= 32 (so at most M blocks of at
// most 32 tokens).
size_t decode_ws_bound(const mla_handle* h, long M) {
  if (h->cfg.dtype != MLA_BF16 || h->lay.H > 32 || h->cfg.page_size % 128) return 0;
  return tc::decode_workspace_bound(h, M, 32);
}

FwdWs forward_ws(const mla_handle* h, long M) {
  const Layout& l = h->lay;
  FwdWs w;
  size_t o = 0;
  w.a_out = o;  o = align256(o + (size_t)M * l.NA * 4);
  w.q_cn = o;   o = align256(o + (size_t)M * l.rq * l.elt);
  w.q_raw = o;  o = align256(o + (l.rq > 0 ? (size_t)M * l.H * l.dqk * 4 : 0));
  w.q_nope = o; o = align256(o + (size_t)M * l.H * l.dn * l.elt);
  w.q_abs = o;  o = align256(o + (size_t)M * l.H * l.L * l.elt);
  w.o_lat = o;  o = align256(o + (size_t)M * l.H * l.rkv * l.elt);
  w.o = o;      o = align256(o + (size_t)M * l.H * l.dv * l.elt);
  w.dec = o;    w.dec_bytes = decode_ws_bound(h, M); o = align256(o + w.dec_bytes);
  w.total = o;
  return w;
}

// The bf16 append runs as one fused kernel when its CTAs (3 per 128 rows)
// fill the GPU; fewer tokens, and the fp32 layer, stage the projection (a
// split-K GEMM) in a workspace and finish the rows with a second kernel.
bool append_fused(const mla_handle* h, long n) {
  return h->cfg.dtype == MLA_BF16 && 3L * ((n + 127) / 128) >= h->num_sms;
}
size_t append_ws(const mla_handle* h, long n) {
  return append_fused(h, n) ? 0 : align256((size_t)n * h->lay.L * 4);
}

}  // namespace
}  // namespace mla

extern "C" size_t mla_append_workspace_bytes(const mla_handle_t* h, int32_t n) {
  return (h && n >= 0) ? append_ws(h, n) : 0;
}

extern "C" size_t mla_forward_workspace_bytes(const mla_handle_t* h, int32_t num_tokens) {
  return (h && num_tokens >= 0) ? forward_ws(h, num_tokens).total : 0;
}

namespace mla {
namespace {
// The expanded form's pieces after the forward's own: the gathered latent
// rows [rows, L] (layer dtype) and their expansion [rows, H, dn + dv] (fp16).
struct SharedWs {
  size_t gathered, kv, units, total;
};
SharedWs shared_ws(const mla_handle* h, long num_tokens, long ctx_rows) {
  const Layout& l = h->lay;
  const long rows = ctx_rows + num_tokens;
  SharedWs w;
  size_t o = forward_ws(h, num_tokens).total;
  w.gathered = o; o = align256(o + (size_t)rows * l.L * l.elt);
  w.kv = o;       o = align256(o + (size_t)rows * l.H * (l.dn + l.dv) * 2);
  w.units = o;    o = align256(o + (size_t)3 * num_tokens * 4);   // >= num_blocks + 2 * num_ctx ints
  w.total = o;
  return w;
}
}  // namespace
}  // namespace mla

extern "C" size_t mla_forward_shared_workspace_bytes(const mla_handle_t* h, int32_t num_tokens,
                                                     int32_t ctx_rows) {
  return (h && num_tokens >= 0 && ctx_rows >= 0) ? shared_ws(h, num_tokens, ctx_rows).total : 0;
}

// ---------------------------------------------------------------------------
// Projections: tcgen05 GEMM for 16-bit operands, SIMT for the fp32 layer
// ---------------------------------------------------------------------------
namespace mla {
namespace {

template <typename TA, typename TC>
mla_status_t proj(mla_handle_t* h, cudaStream_t st, bool pdl, int M, int N, int K, int batch,
                  const TA* A, long lda, long sA, const TA* B, long ldb, long sB, TC* C, long ldc,
                  long sC, const float* G = nullptr, long ldg = 0, long sG = 0, bool gate_act = false,
                  int sig_from = -1, const tc::QSplit* qsplit = nullptr, bool* qsplit_done = nullptr) {
  h->launches += (M > 0 && N > 0 && batch > 0);
  if constexpr (std::is_same<TA, float>::value) {
    simt::gemm_nt<TA, TC>(st, M, N, K, batch, A, lda, sA, B, ldb, sB, C, ldc, sC, G, ldg, sG);
    return MLA_OK;
  } else {
    tc::Out o = std::is_same<TC, float>::value ? tc::Out::F32
                : std::is_same<TC, __half>::value ? tc::Out::F16 : tc::Out::BF16;
    tc::GemmArgs a{M, N, K, batch, std::is_same<TA, __half>::value, A, lda, sA, B, ldb, sB,
                   C, ldc, sC, o, G, ldg, sG, pdl, gate_act, sig_from, qsplit, qsplit_done};
    return tc::gemm(st, a, h->status);
  }
}

}  // namespace
}  // namespace mla

// ---------------------------------------------------------------------------
// Latent-cache append
// ---------------------------------------------------------------------------
namespace mla {
namespace {

template <typename T>
mla_status_t append_impl(mla_handle_t* h, const void* hidden, const int32_t* positions,
                 const int64_t* slots, int n, void* cache, long num_slots, float* kv_ws,
                 cudaStream_t st) {
  const Layout& l = h->lay;
  // kv = hidden @ W_kva^T : W_kva = first L rows of W_A
  if constexpr (std::is_same<T, __nv_bfloat16>::value) {
    if (append_fused(h, n)) {
      h->launches += 1;
      return tc::kv_append(st, h, (const T*)hidden, n, positions, slots, (T*)cache, num_slots,
                           true);
    }
  }
  {
    mla_status_t s = proj<T, float>(h, st, false, n, l.L, l.D, 1, (const T*)hidden, l.D, 0,
                                    (const T*)h->WA, l.D, 0, kv_ws, l.L, 0);
    if (s != MLA_OK) return s;
    simt::kv_finish<T>(st, h, kv_ws, l.L, n, positions, slots, (T*)cache, num_slots);
    h->launches += 1;
    return MLA_OK;
  }
}

}  // namespace
}  // namespace mla

extern "C" mla_status_t mla_latent_cache_append(mla_handle_t* h, const void* hidden,
                                                const int32_t* positions,
                                                const int64_t* slot_mapping, int32_t n,
                                                void* cache, int32_t num_pages, void* workspace,
                                                size_t workspace_bytes, void* stream) {
  if (!h) return fail(MLA_ERR_INVALID_ARG, "append: null handle");
  if (n < 0) return fail(MLA_ERR_INVALID_ARG, "append: n < 0");
  if (n == 0) return MLA_OK;
  if (!hidden || !positions || !slot_mapping || !cache || (!workspace && append_ws(h, n)))
    return fail(MLA_ERR_INVALID_ARG, "append: null pointer");
  if (num_pages <= 0) return fail(MLA_ERR_INVALID_ARG, "append: num_pages <= 0");
  if (workspace_bytes < append_ws(h, n))
    return fail(MLA_ERR_INVALID_ARG, "append: workspace smaller than mla_append_workspace_bytes()");
  cudaStream_t st = (cudaStream_t)stream;
  const long num_slots = (long)num_pages * h->cfg.page_size;
  const mla_status_t s =
      h->cfg.dtype == MLA_BF16
          ? append_impl<__nv_bfloat16>(h, hidden, positions, slot_mapping, n, cache, num_slots,
                                       (float*)workspace, st)
          : append_impl<float>(h, hidden, positions, slot_mapping, n, cache, num_slots,
                               (float*)workspace, st);
  if (s != MLA_OK) return s;
  MLA_CUDA_TRY(cudaGetLastError());
  return MLA_OK;
}

// ---------------------------------------------------------------------------
// Forward
// ---------------------------------------------------------------------------
namespace mla {
namespace {

template <typename TX, typename TI>
mla_status_t forward_impl(mla_handle_t* h, const void* hidden, const int32_t* pos, const int64_t* bslots,
                  void* cache, int num_pages, const mla_attn_desc_t& d, void* out, char* ws,
                  cudaStream_t st, cudaEvent_t kv_ready, const mla_shared_ctx_t* ctx = nullptr) {
  const Layout& l = h->lay;
  const int M = d.num_blocks * d.block_len;
  const FwdWs w = forward_ws(h, M);
  float* a_out = (float*)(ws + w.a_out);
  const TX* x = (const TX*)hidden;
  const TX* WA = (const TX*)h->WA;
  // A projection; the block's own latents only when it writes them.  Enough
  // tokens to fill the GPU with the fused append kernel (3 CTAs per 128 rows):
  // that kernel; fewer tokens (or fp32): the latent rows join the projection
  // (split-K spreads it over the SMs) and the finish kernel normalises,
  // rotates and stores them.
  constexpr bool kBf16 = std::is_same<TX, __nv_bfloat16>::value;
  const long num_slots = (long)num_pages * h->cfg.page_size;
  const bool fused_kv = kBf16 && bslots && 3L * ((M + 127) / 128) >= h->num_sms;
  const int r0 = (bslots && !fused_kv) ? 0 : l.L;
  // every kernel (bf16 layers) may start while the previous kernel of the
  // stream finishes (programmatic dependent launch) and waits for it on the
  // device before it reads anything but the weights; a first kernel behind a
  // copy or an event wait starts as a plain launch
  constexpr bool pdl = kBf16;
  // (tensor-core layers: the gate columns leave this GEMM as sigmoid(x W_gate^T))
  mla_status_t s = proj<TX, float>(h, st, pdl, M, l.NA - r0, l.D, 1, x, l.D, 0,
                                   WA + (long)r0 * l.D, l.D, 0, a_out + r0, l.NA, 0, nullptr, 0, 0,
                                   false, l.gdim ? l.L + l.qdim - r0 : -1);
  if (s != MLA_OK) return s;
  if (bslots) {
    if (fused_kv) {
      if constexpr (kBf16) {
        s = tc::kv_append(st, h, x, M, pos, bslots, (TX*)cache, num_slots, pdl);
        if (s != MLA_OK) return s;
      }
    } else {
      simt::kv_finish<TX>(st, h, a_out, l.NA, M, pos, bslots, (TX*)cache, num_slots, pdl);
    }
  }
  const float* q_raw;
  long ldq;
  TI* q_nope = (TI*)(ws + w.q_nope);
  // Q_abs shares the cache's type: the two meet in the attention contraction
  TX* q_abs = (TX*)(ws + w.q_abs);
  bool split_done = false;
  if (l.rq > 0) {
    TI* q_cn = (TI*)(ws + w.q_cn);
    simt::rmsnorm_rows<TI>(st, a_out + l.L, l.NA, M, l.rq, h->gamma_q, (float)h->cfg.rms_norm_eps, q_cn,
                           pdl);
    float* qr = (float*)(ws + w.q_raw);
    // tensor-core layers: the GEMM's epilogue may split the heads and rotate
    // the RoPE dims itself (persistent launches), else the row kernel below
    tc::QSplit qs{};
    if constexpr (kBf16)
      qs = tc::QSplit{(__half*)q_nope, (__nv_bfloat16*)q_abs, pos, h->rope, l.H, l.dn, l.dr, l.L, l.rkv,
                      h->cfg.max_position, (int)(h->cfg.rope == MLA_ROPE_INTERLEAVED)};
    s = proj<TI, float>(h, st, pdl, M, l.H * l.dqk, l.rq, 1, q_cn, l.rq, 0, (const TI*)h->Wqb, l.rq,
                        0, qr, l.H * l.dqk, 0, nullptr, 0, 0, false, -1, kBf16 ? &qs : nullptr,
                        &split_done);
    if (s != MLA_OK) return s;
    q_raw = qr;
    ldq = l.H * l.dqk;
  } else {
    q_raw = a_out + l.L;
    ldq = l.NA;
  }
  if (!split_done) simt::q_rope_split<TI, TX>(st, h, q_raw, ldq, M, pos, q_nope, q_abs, pdl);
  if constexpr (kBf16) {
    if (ctx && tc::expand_applies(h, d.block_len)) {
      // blocks sharing contexts, the expanded form: each context's latents and
      // each block's own gathered once, expanded by kv_b_proj into per-head
      // k_nope | v, then one attention of q_nope | q_pe over them (its output
      // already o[h], times the gate); no W_UK / W_UV absorption
      if (kv_ready) MLA_CUDA_TRY(cudaStreamWaitEvent(st, kv_ready, 0));
      const SharedWs sw = shared_ws(h, M, ctx->ctx_rows);
      const long rows = tc::expand_rows(*ctx, d.num_blocks, d.block_len);
      TX* gathered = (TX*)(ws + sw.gathered);
      __half* kvx = (__half*)(ws + sw.kv);
      tc::expand_gather(st, h, (const TX*)cache, num_pages, d, *ctx, gathered, pdl && !kv_ready);
      s = proj<TX, TI>(h, st, pdl, rows, l.H * (l.dn + l.dv), l.rkv, 1, gathered, l.L, 0,
                       (const TX*)h->WKV, l.rkv, 0, (TI*)kvx, (long)l.H * (l.dn + l.dv), 0);
      if (s != MLA_OK) return s;
      TI* o = (TI*)(ws + w.o);
      const float* gate = l.gdim ? a_out + l.L + l.qdim : nullptr;
      s = tc::expanded_attention(st, h, (const __half*)q_nope, (const __nv_bfloat16*)q_abs, kvx,
                                 gathered, rows, d, *ctx, pos, gate, l.NA, (__half*)o,
                                 (int32_t*)(ws + sw.units), pdl);
      if (s != MLA_OK) return s;
      s = proj<TI, TX>(h, st, pdl, M, l.D, l.H * l.dv, 1, o, (long)l.H * l.dv, 0, (const TI*)h->Wo,
                       (long)l.H * l.dv, 0, (TX*)out, l.D, 0);
      if (s != MLA_OK) return s;
      // non-GEMM kernels: [kv finish], [q norm], [rope split], gather, [unit
      // order], attention
      h->launches += (split_done ? 2 : 3) + (bslots ? 1 : 0) + (l.rq > 0 ? 1 : 0) +
                     (tc::expand_grouped(d.block_len) ? 1 : 0);
      return MLA_OK;
    }
  }
  // q_lat[h] = q_nope[h] @ W_UK[h]  ->  Q_abs[:, h, :rkv]
  s = proj<TI, TX>(h, st, pdl, M, l.rkv, l.dn, l.H, q_nope, (long)l.H * l.dn, l.dn,
                   (const TI*)h->WUKT, l.dn, (long)l.rkv * l.dn, q_abs, (long)l.H * l.L, l.L);
  if (s != MLA_OK) return s;
  TI* o_lat = (TI*)(ws + w.o_lat);
  // the cache writes of another stream the attention depends on (a plain
  // launch after the wait: no programmatic edge crosses it)
  if (kv_ready) MLA_CUDA_TRY(cudaStreamWaitEvent(st, kv_ready, 0));
  if constexpr (std::is_same<TX, float>::value) {
    simt::latent_attention<TI, TX>(st, h, q_abs, (const TX*)cache, num_pages, d, pos, o_lat);
  } else if (tc::decode_applies(h, d.block_len)) {
    // few query rows per block: keys in the MMA's M dimension, splits merged after
    s = tc::latent_decode(st, h, q_abs, (const TX*)cache, num_pages, d, pos, o_lat, nullptr,
                          ws + w.dec, w.dec_bytes, pdl && !kv_ready);
    if (s != MLA_OK) return s;
    h->launches += 1;     // the merge
  } else {
    s = tc::latent_attention(st, h, q_abs, (const TX*)cache, num_pages, d, pos, o_lat, nullptr,
                             pdl && !kv_ready);
    if (s != MLA_OK) return s;
  }
  // o[h] = o_lat[h] @ W_UV[h]^T (* sigmoid(gate): computed by the A projection on
  // tensor-core layers, by this GEMM's epilogue on the fp32 layer)
  TI* o = (TI*)(ws + w.o);
  const float* gate = l.gdim ? a_out + l.L + l.qdim : nullptr;
  s = proj<TI, TI>(h, st, pdl, M, l.dv, l.rkv, l.H, o_lat, (long)l.H * l.rkv, l.rkv,
                   (const TI*)h->WUV, l.rkv, (long)l.dv * l.rkv, o, (long)l.H * l.dv, l.dv, gate,
                   l.NA, l.dv, kBf16);
  if (s != MLA_OK) return s;
  s = proj<TI, TX>(h, st, pdl, M, l.D, l.H * l.dv, 1, o, (long)l.H * l.dv, 0, (const TI*)h->Wo,
                   (long)l.H * l.dv, 0, (TX*)out, l.D, 0);
  if (s != MLA_OK) return s;
  // non-GEMM kernels: [kv finish], [q norm], [rope split], attention
  h->launches += (split_done ? 1 : 2) + (bslots ? 1 : 0) + (l.rq > 0 ? 1 : 0);
  return MLA_OK;
}

}  // namespace
}  // namespace mla

extern "C" mla_status_t mla_draft_forward_after(mla_handle_t* h, const void* hidden,
                                                const int32_t* positions,
                                                const int64_t* block_slot_mapping, void* cache,
                                                int32_t num_pages, const mla_attn_desc_t* desc,
                                                void* out, void* workspace,
                                                size_t workspace_bytes, void* stream,
                                                void* cache_ready) {
  if (!h || !desc) return fail(MLA_ERR_INVALID_ARG, "forward: null handle or descriptor");
  const mla_attn_desc_t& d = *desc;
  if (d.num_blocks < 0 || d.block_len <= 0 || d.max_pages <= 0)
    return fail(MLA_ERR_INVALID_ARG, "forward: num_blocks >= 0, block_len > 0, max_pages > 0");
  if (d.num_blocks == 0) return MLA_OK;
  if ((long)d.num_blocks * d.block_len > 0x7fffffffL)
    return fail(MLA_ERR_INVALID_ARG, "forward: too many tokens");
  if (!hidden || !positions || !cache || !out || !workspace || !d.block_table || !d.kv_len)
    return fail(MLA_ERR_INVALID_ARG, "forward: null pointer");
  if (num_pages <= 0) return fail(MLA_ERR_INVALID_ARG, "forward: num_pages <= 0");
  const int M = d.num_blocks * d.block_len;
  if (workspace_bytes < forward_ws(h, M).total)
    return fail(MLA_ERR_INVALID_ARG, "forward: workspace smaller than mla_forward_workspace_bytes()");
  if ((uintptr_t)workspace % 256) return fail(MLA_ERR_INVALID_ARG, "forward: workspace must be 256-byte aligned");
  cudaStream_t st = (cudaStream_t)stream;
  const cudaEvent_t ev = (cudaEvent_t)cache_ready;
  const mla_status_t s =
      h->cfg.dtype == MLA_BF16
          ? forward_impl<__nv_bfloat16, __half>(h, hidden, positions, block_slot_mapping, cache,
                                                num_pages, d, out, (char*)workspace, st, ev)
          : forward_impl<float, float>(h, hidden, positions, block_slot_mapping, cache,
                                       num_pages, d, out, (char*)workspace, st, ev);
  if (s != MLA_OK) return s;
  MLA_CUDA_TRY(cudaGetLastError());
  return MLA_OK;
}

extern "C" mla_status_t mla_draft_forward_shared_after(mla_handle_t* h, const void* hidden,
                                                       const int32_t* positions,
                                                       const int64_t* block_slot_mapping, void* cache,
                                                       int32_t num_pages, const mla_attn_desc_t* desc,
                                                       const mla_shared_ctx_t* ctx, void* out,
                                                       void* workspace, size_t workspace_bytes,
                                                       void* stream, void* cache_ready) {
  if (!h || !desc || !ctx) return fail(MLA_ERR_INVALID_ARG, "forward_shared: null handle, descriptor or context list");
  const mla_attn_desc_t& d = *desc;
  if (d.num_blocks < 0 || d.block_len <= 0 || d.max_pages <= 0)
    return fail(MLA_ERR_INVALID_ARG, "forward_shared: num_blocks >= 0, block_len > 0, max_pages > 0");
  if (d.num_blocks == 0) return MLA_OK;
  if (ctx->num_ctx <= 0 || ctx->num_ctx > d.num_blocks || ctx->ctx_rows < 0 || !ctx->ctx_len || !ctx->ctx_block_start)
    return fail(MLA_ERR_INVALID_ARG,
                "forward_shared: 0 < num_ctx <= num_blocks, ctx_rows >= 0, ctx_len and ctx_block_start set");
  if ((long)d.num_blocks * d.block_len + ctx->ctx_rows > 0x7fffffffL)
    return fail(MLA_ERR_INVALID_ARG, "forward_shared: too many tokens");
  if (!hidden || !positions || !cache || !out || !workspace || !d.block_table || !d.kv_len)
    return fail(MLA_ERR_INVALID_ARG, "forward_shared: null pointer");
  if (num_pages <= 0) return fail(MLA_ERR_INVALID_ARG, "forward_shared: num_pages <= 0");
  const int M = d.num_blocks * d.block_len;
  if (workspace_bytes < shared_ws(h, M, ctx->ctx_rows).total)
    return fail(MLA_ERR_INVALID_ARG, "forward_shared: workspace smaller than mla_forward_shared_workspace_bytes()");
  if ((uintptr_t)workspace % 256) return fail(MLA_ERR_INVALID_ARG, "forward_shared: workspace must be 256-byte aligned");
  cudaStream_t st = (cudaStream_t)stream;
  const cudaEvent_t ev = (cudaEvent_t)cache_ready;
  const mla_status_t s =
      h->cfg.dtype == MLA_BF16
          ? forward_impl<__nv_bfloat16, __half>(h, hidden, positions, block_slot_mapping, cache,
                                                num_pages, d, out, (char*)workspace, st, ev, ctx)
          : forward_impl<float, float>(h, hidden, positions, block_slot_mapping, cache,
                                       num_pages, d, out, (char*)workspace, st, ev);
  if (s != MLA_OK) return s;
  MLA_CUDA_TRY(cudaGetLastError());
  return MLA_OK;
}

extern "C" mla_status_t mla_draft_forward_shared(mla_handle_t* h, const void* hidden,
                                                 const int32_t* positions,
                                                 const int64_t* block_slot_mapping, void* cache,
                                                 int32_t num_pages, const mla_attn_desc_t* desc,
                                                 const mla_shared_ctx_t* ctx, void* out,
                                                 void* workspace, size_t workspace_bytes,
                                                 void* stream) {
  return mla_draft_forward_shared_after(h, hidden, positions, block_slot_mapping, cache, num_pages,
                                        desc, ctx, out, workspace, workspace_bytes, stream, nullptr);
}

extern "C" mla_status_t mla_shared_attention(mla_handle_t* h, const int32_t* positions,
                                             const mla_attn_desc_t* desc, const mla_shared_ctx_t* ctx,
                                             void* workspace, size_t workspace_bytes, void* stream) {
  if (!h || !desc || !ctx || !positions || !workspace)
    return fail(MLA_ERR_INVALID_ARG, "shared_attention: null pointer");
  const mla_attn_desc_t& d = *desc;
  if (d.num_blocks <= 0 || d.block_len <= 0 || ctx->num_ctx <= 0 || ctx->num_ctx > d.num_blocks ||
      ctx->ctx_rows < 0 || !ctx->ctx_len || !ctx->ctx_block_start)
    return fail(MLA_ERR_INVALID_ARG,
                "shared_attention: num_blocks, block_len > 0, 0 < num_ctx <= num_blocks, ctx_rows >= 0");
  if (!tc::expand_applies(h, d.block_len))
    return fail(MLA_ERR_UNSUPPORTED, "shared_attention: the layer does not run the expanded form");
  const Layout& l = h->lay;
  const long M = (long)d.num_blocks * d.block_len;
  const SharedWs sw = shared_ws(h, M, ctx->ctx_rows);
  if (workspace_bytes < sw.total)
    return fail(MLA_ERR_INVALID_ARG, "shared_attention: workspace smaller than mla_forward_shared_workspace_bytes()");
  const FwdWs w = forward_ws(h, M);
  char* ws = (char*)workspace;
  const float* gate = l.gdim ? (const float*)(ws + w.a_out) + l.L + l.qdim : nullptr;
  const mla_status_t s = tc::expanded_attention(
      (cudaStream_t)stream, h, (const __half*)(ws + w.q_nope), (const __nv_bfloat16*)(ws + w.q_abs),
      (const __half*)(ws + sw.kv), (const __nv_bfloat16*)(ws + sw.gathered),
      tc::expand_rows(*ctx, d.num_blocks, d.block_len), d, *ctx, positions, gate, l.NA,
      (__half*)(ws + w.o), (int32_t*)(ws + sw.units), false);
  if (s != MLA_OK) return s;
  MLA_CUDA_TRY(cudaGetLastError());
  return MLA_OK;
}

extern "C" mla_status_t mla_draft_forward(mla_handle_t* h, const void* hidden,
                                          const int32_t* positions,
                                          const int64_t* block_slot_mapping, void* cache,
                                          int32_t num_pages, const mla_attn_desc_t* desc,
                                          void* out, void* workspace, size_t workspace_bytes,
                                          void* stream) {
  return mla_draft_forward_after(h, hidden, positions, block_slot_mapping, cache, num_pages, desc,
                                 out, workspace, workspace_bytes, stream, nullptr);
}

extern "C" size_t mla_forward_workspace_offset(const mla_handle_t* h, int32_t num_tokens,
                                               int32_t part) {
  if (!h || num_tokens < 0) return (size_t)-1;
  const FwdWs w = forward_ws(h, num_tokens);
  switch (part) {
    case MLA_WS_Q_ABS: return w.q_abs;
    case MLA_WS_O_LAT: return w.o_lat;
    case MLA_WS_O: return w.o;
    default: return (size_t)-1;
  }
}

extern "C" size_t mla_latent_attention_workspace_bytes(const mla_handle_t* h,
                                                      const mla_attn_desc_t* desc) {
  if (!h || !desc || desc->num_blocks <= 0 || desc->block_len <= 0 || desc->max_pages <= 0) return 0;
  return tc::decode_applies(h, desc->block_len) ? tc::decode_workspace_bytes(h, *desc) : 0;
}

extern "C" mla_status_t mla_latent_attention(mla_handle_t* h, const void* q_abs,
                                             const int32_t* positions, const void* cache,
                                             int32_t num_pages, const mla_attn_desc_t* desc,
                                             void* o_lat, float* lse, void* workspace,
                                             size_t workspace_bytes, void* stream) {
  if (!h || !desc) return fail(MLA_ERR_INVALID_ARG, "attention: null handle or descriptor");
  const mla_attn_desc_t& d = *desc;
  if (d.num_blocks < 0 || d.block_len <= 0 || d.max_pages <= 0)
    return fail(MLA_ERR_INVALID_ARG, "attention: num_blocks >= 0, block_len > 0, max_pages > 0");
  if (d.num_blocks == 0) return MLA_OK;
  if ((long)d.num_blocks * d.block_len * h->lay.H > 0x7fffffffL)
    return fail(MLA_ERR_INVALID_ARG, "attention: too many rows");
  if (!q_abs || !positions || !cache || !o_lat || !d.block_table || !d.kv_len)
    return fail(MLA_ERR_INVALID_ARG, "attention: null pointer");
  if (num_pages <= 0) return fail(MLA_ERR_INVALID_ARG, "attention: num_pages <= 0");
  if ((uintptr_t)q_abs % 16 || (uintptr_t)o_lat % 16 || (uintptr_t)cache % 16)
    return fail(MLA_ERR_INVALID_ARG, "attention: q_abs, cache and o_lat must be 16-byte aligned");
  cudaStream_t st = (cudaStream_t)stream;
  h->launches += 1;
  if (h->cfg.dtype == MLA_BF16 && tc::decode_applies(h, d.block_len)) {
    const size_t need = tc::decode_workspace_bytes(h, d);
    if (!workspace || workspace_bytes < need || (uintptr_t)workspace % 256)
      return fail(MLA_ERR_INVALID_ARG,
                  "attention: workspace smaller than mla_latent_attention_workspace_bytes() or not 256-byte aligned");
    const mla_status_t s = tc::latent_decode(st, h, (const __nv_bfloat16*)q_abs,
                                             (const __nv_bfloat16*)cache, num_pages, d, positions,
                                             (__half*)o_lat, lse, workspace, workspace_bytes, false);
    if (s != MLA_OK) return s;
    h->launches += 1;
  } else if (h->cfg.dtype == MLA_BF16) {
    const mla_status_t s = tc::latent_attention(st, h, (const __nv_bfloat16*)q_abs,
                                                (const __nv_bfloat16*)cache, num_pages, d,
                                                positions, (__half*)o_lat, lse, false);
    if (s != MLA_OK) return s;
  } else {
    simt::latent_attention<float, float>(st, h, (const float*)q_abs, (const float*)cache,
                                         num_pages, d, positions, (float*)o_lat, lse);
  }
  MLA_CUDA_TRY(cudaGetLastError());
  return MLA_OK;
}

extern "C" mla_status_t mla_get_device_status(mla_handle_t* h, void* stream, int32_t* bits) {
  if (!h) return fail(MLA_ERR_INVALID_ARG, "status: null handle");
  cudaStream_t st = (cudaStream_t)stream;
  uint32_t v = 0;
  MLA_CUDA_TRY(cudaStreamSynchronize(st));
  MLA_CUDA_TRY(cudaMemcpy(&v, h->status, sizeof(v), cudaMemcpyDeviceToHost));
  MLA_CUDA_TRY(cudaMemset(h->status, 0, sizeof(v)));
  if (bits) *bits = (int32_t)v;
  if (v & MLA_DEV_TIMEOUT) return fail(MLA_ERR_TIMEOUT, "device: a bounded wait expired");
  if (v) return fail(MLA_ERR_DEVICE_CHECK, "device: index check failed (bits " + std::to_string(v) + ")");
  return MLA_OK;
}

extern "C" unsigned long long mla_kernel_launches(const mla_handle_t* h) { return h ? h->launches : 0; }
