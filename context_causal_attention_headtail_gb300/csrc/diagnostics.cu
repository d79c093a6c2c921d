// Diagnostic kernel for the bounded waits: one thread waits, through the same
// mbar_wait the attention kernels use, on an mbarrier that nothing arrives
// at. The wait gives up after the given limit, raises the CTA's abort flag and
// ERR_FLAG_TIMEOUT on the device error flag, and the kernel returns. Nothing
// else is in flight (no TMA copy, no MMA, no tensor memory), so the context
// stays usable and the next call works as before.
#include "tc_common.cuh"

namespace cpattn {
namespace {

__global__ void __launch_bounds__(32, 1) wait_probe_kernel(int *err, unsigned long long limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x != 0) return;
  abort_flag = 0;
  const uint32_t b = tc::smem_u32(&bar);
  tc::mbar_init(b, 1);
  tc::mbar_fence_init();
  const tc::WaitCtx w{&abort_flag, err, limit_ns};
  tc::mbar_wait(b, 0, w);   // phase 0 never completes: no thread arrives
}

}  // namespace

cpattn_status launch_wait_probe(unsigned long long limit_ns, cudaStream_t s) {
  int *err = device_err_flag();
  if (!err) return fail(CPATTN_ERR_CUDA, "cannot resolve the device error flag");
  wait_probe_kernel<<<1, 32, 0, s>>>(err, limit_ns);
  return check_launch("wait probe kernel");
}

}  // namespace cpattn
