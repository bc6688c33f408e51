// status.cu — status strings and the device status read-back.
#include <cuda_runtime.h>

#include "rl_device.cuh"

extern "C" const char* rl_status_string(rl_status status) {
  switch (status) {
    case RL_OK: return "ok";
    case RL_ERR_NULL: return "a required pointer is NULL";
    case RL_ERR_SHAPE: return "a size is out of range";
    case RL_ERR_DTYPE: return "unknown element type or advantage layout";
    case RL_ERR_ALIGN: return "logits/dlogits base or row stride not 16-byte aligned";
    case RL_ERR_ALIAS: return "dlogits partially overlaps logits";
    case RL_ERR_WORKSPACE: return "workspace missing or too small";
    case RL_ERR_ID_RANGE: return "a sampled id is outside [0, V) on a valid token";
    case RL_ERR_TIMEOUT: return "a bounded on-chip wait timed out";
    case RL_ERR_CUDA: return "a CUDA runtime call or launch failed";
    case RL_ERR_ARG: return "a scalar argument is out of range";
  }
  return "unknown status";
}

extern "C" rl_status rl_read_device_status(const void* workspace, void* stream) {
  if (!workspace) return RL_ERR_NULL;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return RL_ERR_CUDA;
  unsigned int word = 0;
  const auto* hdr = static_cast<const rl::WsHeader*>(workspace);
  if (cudaMemcpy(&word, &hdr->last_status, sizeof word, cudaMemcpyDeviceToHost) != cudaSuccess)
    return RL_ERR_CUDA;
  if (word & RL_DEVERR_ID_RANGE) return RL_ERR_ID_RANGE;
  if (word & RL_DEVERR_TIMEOUT) return RL_ERR_TIMEOUT;
  return RL_OK;
}

// ------------------------------------------------------------------ wait self-test
namespace rl {
namespace {

// One thread waits on a shared-memory barrier that nothing ever completes,
// through the same bounded wait the kernels use, then reports.
__global__ void wait_selftest_kernel(unsigned long long limit_ns, unsigned int* status,
                                     unsigned long long* waited_ns) {
  __shared__ unsigned long long bar;
  __shared__ int abort;
  if (threadIdx.x != 0) return;
  abort = 0;
  mbar_init(smem_addr(&bar), 1);
  fence_mbar_init();
  const uint64_t t0 = global_ns();
  const bool ok = wait_bounded_for<false>(smem_addr(&bar), 0, &abort, limit_ns);
  const uint64_t t1 = global_ns();
  if (!ok) atomicOr(status, RL_DEVERR_TIMEOUT);
  if (waited_ns) *waited_ns = t1 - t0;
}

}  // namespace
}  // namespace rl

extern "C" rl_status rl_selftest_wait_timeout(unsigned long long limit_ns, unsigned int* status_dev,
                                              unsigned long long* waited_ns_dev, void* stream) {
  if (!status_dev) return RL_ERR_NULL;
  if (limit_ns < 1000ull || limit_ns > 10ull * 1000ull * 1000ull * 1000ull) return RL_ERR_ARG;
  rl::wait_selftest_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(limit_ns, status_dev,
                                                                           waited_ns_dev);
  return cudaGetLastError() == cudaSuccess ? RL_OK : RL_ERR_CUDA;
}
