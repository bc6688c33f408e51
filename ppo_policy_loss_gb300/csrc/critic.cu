// critic.cu — rl_value_loss_fwd_bwd: the PPO clipped value (critic) loss and
// its gradient with respect to the values (sm_103a).
//
// The pages give the PPO loop an actor and a critic (ainews.cool RL.cu
// article, section "技术深度解析", actor/critic bullet); this is the critic's
// half of the update.  O(n) bytes, so one CTA of 1024 threads: a pass that
// counts the valid tokens, then a pass that writes the gradient and reduces
// the loss in fp64 in a fixed order (deterministic).
#include <cmath>

#include "rl_device.cuh"

namespace rl {
namespace {

constexpr int kThreadsV = 1024;
constexpr int kWarpsV = kThreadsV / 32;
constexpr int kUnrollV = 8;

template <typename T>
__device__ __forceinline__ T warp_sum_t(T v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__global__ void __launch_bounds__(kThreadsV, 1)
value_loss_kernel(const float* __restrict__ v, const float* __restrict__ vo,
                  const float* __restrict__ ret, const unsigned char* __restrict__ mask, long long n,
                  float clip, int use_clip, float grad_scale, float* dv, rl_value_stats* stats) {
  __shared__ long long s_cnt[kWarpsV];
  __shared__ double s_red[kWarpsV][3];
  __shared__ long long s_clip[kWarpsV];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // Each step handles kUnrollV tokens per thread, all loaded before any is
  // used; per token the arithmetic is fp32, and only the step sums are added
  // in fp64 (fp64 units are scarce on this GPU).
  constexpr long long kStep = static_cast<long long>(kThreadsV) * kUnrollV;
  long long cnt = 0;
  for (long long i0 = tid; i0 < n; i0 += kStep) {
    unsigned char mv[kUnrollV];
#pragma unroll
    for (int k = 0; k < kUnrollV; ++k) {
      const long long i = i0 + static_cast<long long>(k) * kThreadsV;
      mv[k] = i < n ? mask[i] : 0;
    }
#pragma unroll
    for (int k = 0; k < kUnrollV; ++k) cnt += mv[k] != 0;
  }
  cnt = warp_sum_t(cnt);
  if (lane == 0) s_cnt[warp] = cnt;
  __syncthreads();
  long long N = 0;
  for (int w = 0; w < kWarpsV; ++w) N += s_cnt[w];
  const double inv = N > 0 ? 1.0 / static_cast<double>(N) : 0.0;
  const float scale = static_cast<float>(static_cast<double>(grad_scale) * inv);

  double sumL = 0.0, sumAbs = 0.0;
  long long nclip = 0;
  for (long long i0 = tid; i0 < n; i0 += kStep) {
    unsigned char mv[kUnrollV];
    float vv[kUnrollV], rv[kUnrollV], ov[kUnrollV];
#pragma unroll
    for (int k = 0; k < kUnrollV; ++k) {
      const long long i = i0 + static_cast<long long>(k) * kThreadsV;
      const bool in = i < n;
      mv[k] = in ? mask[i] : 0;
      vv[k] = in ? v[i] : 0.f;
      rv[k] = in ? ret[i] : 0.f;
      ov[k] = in && use_clip ? vo[i] : 0.f;
    }
    float l8 = 0.f, a8 = 0.f;  // this step's terms in fp32; the step sums go to fp64
#pragma unroll
    for (int k = 0; k < kUnrollV; ++k) {
      const long long i = i0 + static_cast<long long>(k) * kThreadsV;
      if (i >= n) continue;
      if (!mv[k]) {
        if (dv) dv[i] = 0.f;
        continue;
      }
      const float d = vv[k] - rv[k];
      const float u = d * d;
      float g = d, L2 = u;
      if (use_clip) {
        const float delta = vv[k] - ov[k];
        const float dc = (ov[k] + fminf(fmaxf(delta, -clip), clip)) - rv[k];
        const float c = dc * dc;
        if (c > u) {  // the clipped square is the larger: its branch, flat outside the clip
          g = fabsf(delta) <= clip ? dc : 0.f;
          L2 = c;
          ++nclip;
        }
      }
      l8 += 0.5f * L2;
      a8 += fabsf(d);
      if (dv) dv[i] = scale * g;
    }
    sumL += static_cast<double>(l8);
    sumAbs += static_cast<double>(a8);
  }
  sumL = warp_sum_t(sumL);
  sumAbs = warp_sum_t(sumAbs);
  nclip = warp_sum_t(nclip);
  if (lane == 0) {
    s_red[warp][0] = sumL;
    s_red[warp][1] = sumAbs;
    s_clip[warp] = nclip;
  }
  __syncthreads();
  if (tid == 0) {
    double L = 0.0, A = 0.0;
    long long C = 0;
    for (int w = 0; w < kWarpsV; ++w) {
      L += s_red[w][0];
      A += s_red[w][1];
      C += s_clip[w];
    }
    rl_value_stats out;
    out.loss = L * inv;
    out.clip_frac = static_cast<double>(C) * inv;
    out.mean_abs_err = A * inv;
    out.n_tokens = N;
    out.n_clipped = C;
    *stats = out;
  }
}

}  // namespace
}  // namespace rl

extern "C" rl_status rl_value_loss_fwd_bwd(const float* values, const float* values_old,
                                           const float* returns, const unsigned char* mask,
                                           long long n, float clip_eps, float grad_scale,
                                           float* dvalues, rl_value_stats* stats_dev,
                                           void* stream) {
  if (n < 0) return RL_ERR_SHAPE;
  if (!stats_dev) return RL_ERR_NULL;
  if (n > 0 && (!values || !returns || !mask)) return RL_ERR_NULL;
  if (!std::isfinite(grad_scale) || std::isnan(clip_eps)) return RL_ERR_ARG;
  const int use_clip = values_old != nullptr && clip_eps >= 0.f && std::isfinite(clip_eps);
  rl::value_loss_kernel<<<1, rl::kThreadsV, 0, static_cast<cudaStream_t>(stream)>>>(
      values, values_old, returns, mask, n, clip_eps, use_clip, grad_scale, dvalues, stats_dev);
  return cudaGetLastError() == cudaSuccess ? RL_OK : RL_ERR_CUDA;
}
