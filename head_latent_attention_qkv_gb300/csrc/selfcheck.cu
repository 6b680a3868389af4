// Self-check of the library's failure path: a bounded wait that runs out.
//
// Every wait of the library's kernels is bounded (mbar_wait in tc_ptx.cuh):
// when its budget of try_wait rounds runs out it sets MLA_DEV_TIMEOUT in the
// handle's device status word and the kernel returns instead of spinning.
// This entry point exercises exactly that primitive on a barrier that nothing
// will ever arrive on, so that the failure path can be tested without
// faulting or hanging a GPU: one CTA of one thread, no copies, no tensor
// memory, nothing left in flight when it returns.
#include "common.cuh"
#include "tc_ptx.cuh"

namespace {

__global__ void wait_never_armed_kernel(uint32_t* status, uint32_t budget, int32_t* waited) {
  __shared__ uint64_t bar;
  mla::tc::mbar_init(&bar, 1);             // one arrival expected; none will come
  mla::tc::fence_mbar_init();
  const bool ok = mla::tc::mbar_wait(&bar, 0, status, budget);
  *waited = ok ? 0 : 1;
}

}  // namespace

extern "C" mla_status_t mla_check_wait_timeout(mla_handle_t* h, uint32_t max_rounds,
                                               int32_t* gave_up, void* stream) {
  using namespace mla;
  if (!h || !gave_up) return fail(MLA_ERR_INVALID_ARG, "check_wait_timeout: null argument");
  if (max_rounds == 0 || max_rounds > (1u << 24))
    return fail(MLA_ERR_INVALID_ARG, "check_wait_timeout: max_rounds must be in [1, 2^24]");
  cudaStream_t st = (cudaStream_t)stream;
  h->launches += 1;
  wait_never_armed_kernel<<<1, 1, 0, st>>>(h->status, max_rounds, gave_up);
  MLA_CUDA_TRY(cudaGetLastError());
  return MLA_OK;
}
