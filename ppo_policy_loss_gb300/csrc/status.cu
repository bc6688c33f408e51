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
