// advantages.cu — rl_group_advantages and rl_gae_reverse_scan (sm_103a).
//
// The RL.cu pages name reward normalisation (ainews.cool RL.cu article, the
// paragraph after its benchmark table) for GRPO, the group-relative method of
// the pitchhut.com listing ("Key Features" item 3), and advantage estimation
// inside the PPO update (same article, "PPO 更新内核" bullet).  Both steps
// touch O(B*T) bytes, so they are latency kernels: one warp per group, one
// CTA per sequence, fp64 arithmetic (cheap at this size, and exact enough that the
// result is the fp64 definition rounded once to fp32).
#include <cmath>

#include "rl_device.cuh"

namespace rl {
namespace {

constexpr int kWarpsPerBlock = 8;

__device__ __forceinline__ double warp_sum(double v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// One warp per group: two-pass mean and standard deviation, then
// A = (R - mean) / (std + std_eps).
__global__ void __launch_bounds__(kWarpsPerBlock * 32)
group_advantages_kernel(const float* rewards, int n_groups, int G, double std_eps,
                        int ddof, float* adv) {
  allow_dependents();  // the loss launch may start its set-up beside this kernel
  const int gw = blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (gw >= n_groups) return;
  const float* r = rewards + static_cast<long long>(gw) * G;
  double sum = 0.0;
  for (int j = lane; j < G; j += 32) sum += static_cast<double>(r[j]);
  const double mean = warp_sum(sum) / G;
  double sq = 0.0;
  for (int j = lane; j < G; j += 32) {
    const double d = static_cast<double>(r[j]) - mean;
    sq += d * d;
  }
  const double std = sqrt(warp_sum(sq) / (G - ddof));
  const double inv = 1.0 / (std + std_eps);
  // Every index is read and written by the same lane, after the reductions
  // above have consumed all reads, so adv may alias rewards.
  float* a = adv + static_cast<long long>(gw) * G;
  for (int j = lane; j < G; j += 32) a[j] = static_cast<float>((static_cast<double>(r[j]) - mean) * inv);
}

// One CTA of kThreadsG threads per sequence.  Thread k owns the contiguous
// time chunk [k*cs, min(L, (k+1)*cs)).  Each thread folds its chunk into an
// affine map A_start = P + Q * A_after_chunk (Q = c^len, c = gamma*lam); a
// suffix composition of these maps (shuffles inside each warp, then the warp
// totals in order) gives every chunk its incoming A; a second pass over the
// chunk writes A and ret.  The terminal bootstrap is 0:
// delta_{L-1} = r_{L-1} - v_{L-1}.
constexpr int kThreadsG = 256;

__global__ void __launch_bounds__(kThreadsG)
gae_kernel(const float* __restrict__ rewards, const float* __restrict__ values,
           const int* __restrict__ lengths, int B, int T, double gamma, double lam, float* adv,
           float* ret) {
  __shared__ double s_p[kThreadsG / 32], s_q[kThreadsG / 32], s_in[kThreadsG / 32];
  allow_dependents();  // a following loss launch may start its set-up
  const int b = blockIdx.x;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const long long base = static_cast<long long>(b) * T;
  int L = lengths[b];
  L = L < 0 ? 0 : (L > T ? T : L);
  const double c = gamma * lam;
  const int cs = (L + kThreadsG - 1) / kThreadsG;
  const int t0 = min(L, tid * cs), t1 = min(L, t0 + cs);

  auto delta = [&](int t) -> double {
    const double vn = (t + 1 < L) ? static_cast<double>(values[base + t + 1]) : 0.0;
    return static_cast<double>(rewards[base + t]) + gamma * vn - static_cast<double>(values[base + t]);
  };

  double P = 0.0, Q = 1.0;
  for (int t = t1 - 1; t >= t0; --t) {
    P = delta(t) + c * P;
    Q = c * Q;
  }
  // inclusive suffix composition inside the warp: lane l ends with F_l o ... o F_31
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const double P2 = __shfl_down_sync(0xffffffffu, P, o);
    const double Q2 = __shfl_down_sync(0xffffffffu, Q, o);
    if (lane + o < 32) {
      P = P + Q * P2;
      Q = Q * Q2;
    }
  }
  if (lane == 0) {
    s_p[warp] = P;
    s_q[warp] = Q;
  }
  __syncthreads();
  if (tid == 0) {  // A entering each warp's region from the warps after it
    double a = 0.0;
    for (int w = kThreadsG / 32 - 1; w >= 0; --w) {
      s_in[w] = a;
      a = s_p[w] + s_q[w] * a;
    }
  }
  __syncthreads();
  // A at the start of the next thread's chunk: lanes l+1..31 composed, applied
  // to the A entering this warp's region from the warps after it
  double Pn = __shfl_down_sync(0xffffffffu, P, 1), Qn = __shfl_down_sync(0xffffffffu, Q, 1);
  if (lane == 31) {
    Pn = 0.0;
    Qn = 1.0;
  }
  // second pass: outputs
  double a = Pn + Qn * s_in[warp];
  for (int t = t1 - 1; t >= t0; --t) {
    a = delta(t) + c * a;
    adv[base + t] = static_cast<float>(a);
    if (ret) ret[base + t] = static_cast<float>(a + static_cast<double>(values[base + t]));
  }
  for (int t = L + tid; t < T; t += kThreadsG) {
    adv[base + t] = 0.f;
    if (ret) ret[base + t] = 0.f;
  }
}

}  // namespace
}  // namespace rl

using namespace rl;

extern "C" rl_status rl_group_advantages(const float* rewards, int n_groups, int group_size,
                                         double std_eps, int ddof, float* adv_out, void* stream) {
  if (n_groups < 0 || group_size < 1) return RL_ERR_SHAPE;
  if (ddof != 0 && ddof != 1) return RL_ERR_ARG;
  if (!(std_eps >= 0.0) || !std::isfinite(std_eps)) return RL_ERR_ARG;
  if (group_size <= ddof) return RL_ERR_SHAPE;
  if (n_groups == 0) return RL_OK;
  if (!rewards || !adv_out) return RL_ERR_NULL;
  const int blocks = (n_groups + kWarpsPerBlock - 1) / kWarpsPerBlock;
  group_advantages_kernel<<<blocks, kWarpsPerBlock * 32, 0, static_cast<cudaStream_t>(stream)>>>(
      rewards, n_groups, group_size, std_eps, ddof, adv_out);
  return cudaGetLastError() == cudaSuccess ? RL_OK : RL_ERR_CUDA;
}

extern "C" rl_status rl_gae_reverse_scan(const float* rewards, const float* values,
                                         const int* lengths, int B, int T, float gamma, float lam,
                                         float* adv_out, float* returns_out, void* stream) {
  if (B < 0 || T < 0) return RL_ERR_SHAPE;
  if (!std::isfinite(gamma) || !std::isfinite(lam)) return RL_ERR_ARG;
  if (B == 0 || T == 0) return RL_OK;
  if (!rewards || !values || !lengths || !adv_out) return RL_ERR_NULL;
  gae_kernel<<<B, kThreadsG, 0, static_cast<cudaStream_t>(stream)>>>(
      rewards, values, lengths, B, T, static_cast<double>(gamma), static_cast<double>(lam), adv_out,
      returns_out);
  return cudaGetLastError() == cudaSuccess ? RL_OK : RL_ERR_CUDA;
}

// ------------------------------------------------------------------ masked whitening
namespace rl {
namespace {

constexpr int kThreadsW = 1024;

// One CTA: fp64 masked mean, unbiased variance, then (x - mu) / sqrt(var + eps)
// (or x / sqrt(var + eps)); every element is read and written by the same
// thread after the reductions, so out may alias x.  Each pass handles
// kUnrollW elements per thread per step, loaded before any is used.  Per
// element the arithmetic is fp32 (a step's 8 terms summed in fp32, the step
// sums accumulated in fp64): fp64 units are scarce on this GPU, and one CTA
// doing fp64 per element took ~100 us for 32K elements.
constexpr int kUnrollW = 8;

__global__ void __launch_bounds__(kThreadsW, 1)
masked_whiten_kernel(const float* x, const unsigned char* __restrict__ mask, long long n,
                     double eps, int shift_mean, float* out) {
  __shared__ double s_red[kThreadsW / 32][2];
  __shared__ double s_mu, s_inv;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  allow_dependents();  // a following loss launch may start its set-up
  constexpr long long kStep = static_cast<long long>(kThreadsW) * kUnrollW;
  double sum = 0.0, cnt = 0.0;
  for (long long i0 = tid; i0 < n; i0 += kStep) {
    float xv[kUnrollW];
    bool mv[kUnrollW];
#pragma unroll
    for (int k = 0; k < kUnrollW; ++k) {
      const long long i = i0 + static_cast<long long>(k) * kThreadsW;
      mv[k] = i < n && mask[i] != 0;
      xv[k] = i < n ? x[i] : 0.f;
    }
    float s8 = 0.f;
    int c8 = 0;
#pragma unroll
    for (int k = 0; k < kUnrollW; ++k)
      if (mv[k]) {
        s8 += xv[k];
        ++c8;
      }
    sum += static_cast<double>(s8);
    cnt += static_cast<double>(c8);
  }
  sum = warp_sum(sum);
  cnt = warp_sum(cnt);
  if (lane == 0) {
    s_red[warp][0] = sum;
    s_red[warp][1] = cnt;
  }
  __syncthreads();
  if (tid == 0) {
    double S = 0.0, C = 0.0;
    for (int w = 0; w < kThreadsW / 32; ++w) {
      S += s_red[w][0];
      C += s_red[w][1];
    }
    s_mu = C > 0.0 ? S / C : 0.0;
    s_inv = C;  // count, until the variance is known
  }
  __syncthreads();
  const double mu = s_mu, N = s_inv;
  const float mu_f = static_cast<float>(mu);
  double sq = 0.0;
  for (long long i0 = tid; i0 < n; i0 += kStep) {
    float xv[kUnrollW];
    bool mv[kUnrollW];
#pragma unroll
    for (int k = 0; k < kUnrollW; ++k) {
      const long long i = i0 + static_cast<long long>(k) * kThreadsW;
      mv[k] = i < n && mask[i] != 0;
      xv[k] = i < n ? x[i] : 0.f;
    }
    float q8 = 0.f;
#pragma unroll
    for (int k = 0; k < kUnrollW; ++k)
      if (mv[k]) {
        const float d = xv[k] - mu_f;
        q8 = fmaf(d, d, q8);
      }
    sq += static_cast<double>(q8);
  }
  sq = warp_sum(sq);
  __syncthreads();
  if (lane == 0) s_red[warp][0] = sq;
  __syncthreads();
  if (tid == 0) {
    double Q = 0.0;
    for (int w = 0; w < kThreadsW / 32; ++w) Q += s_red[w][0];
    const double var = N > 1.0 ? Q / (N - 1.0) : 0.0;
    s_inv = 1.0 / sqrt(var + eps);
  }
  __syncthreads();
  const float inv = static_cast<float>(s_inv), shift = shift_mean ? mu_f : 0.f;
  for (long long i0 = tid; i0 < n; i0 += kStep) {
    float xv[kUnrollW];
    bool mv[kUnrollW];
#pragma unroll
    for (int k = 0; k < kUnrollW; ++k) {
      const long long i = i0 + static_cast<long long>(k) * kThreadsW;
      mv[k] = i < n && mask[i] != 0;
      xv[k] = i < n ? x[i] : 0.f;
    }
#pragma unroll
    for (int k = 0; k < kUnrollW; ++k) {
      const long long i = i0 + static_cast<long long>(k) * kThreadsW;
      if (i < n) out[i] = mv[k] ? (xv[k] - shift) * inv : 0.f;
    }
  }
}

}  // namespace
}  // namespace rl

extern "C" rl_status rl_masked_whiten(const float* x, const unsigned char* mask, long long n,
                                      double eps, int shift_mean, float* out, void* stream) {
  if (n < 0) return RL_ERR_SHAPE;
  if (!(eps >= 0.0) || !std::isfinite(eps)) return RL_ERR_ARG;
  if (n == 0) return RL_OK;
  if (!x || !mask || !out) return RL_ERR_NULL;
  rl::masked_whiten_kernel<<<1, rl::kThreadsW, 0, static_cast<cudaStream_t>(stream)>>>(
      x, mask, n, eps, shift_mean, out);
  return cudaGetLastError() == cudaSuccess ? RL_OK : RL_ERR_CUDA;
}

// ------------------------------------------------------------------ token counts
namespace rl {
namespace {

constexpr int kThreadsC = 1024;

// One CTA: N = nonzero mask bytes, B' = sequences (rows of T) with any.
__global__ void __launch_bounds__(kThreadsC, 1)
count_tokens_kernel(const unsigned char* __restrict__ mask, long long B, long long T,
                    long long* counts) {
  __shared__ long long s_n[kThreadsC / 32], s_b[kThreadsC / 32];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  allow_dependents();  // a following loss launch may start its set-up
  long long n = 0, nb = 0;
  for (long long b = warp; b < B; b += kThreadsC / 32) {
    long long c = 0;
    for (long long t = lane; t < T; t += 32) c += mask[b * T + t] != 0;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
    n += c;
    nb += c > 0;
  }
  if (lane == 0) {
    s_n[warp] = n;
    s_b[warp] = nb;
  }
  __syncthreads();
  if (tid == 0) {
    long long N = 0, Bp = 0;
    for (int w = 0; w < kThreadsC / 32; ++w) {
      N += s_n[w];
      Bp += s_b[w];
    }
    counts[0] = N;
    counts[1] = Bp;
  }
}

}  // namespace
}  // namespace rl

extern "C" rl_status rl_count_tokens(const unsigned char* mask, long long B, long long T,
                                     long long* counts_dev, void* stream) {
  if (B < 0 || T < 0) return RL_ERR_SHAPE;
  if (!counts_dev || (B * T > 0 && !mask)) return RL_ERR_NULL;
  rl::count_tokens_kernel<<<1, rl::kThreadsC, 0, static_cast<cudaStream_t>(stream)>>>(mask, B, T,
                                                                                     counts_dev);
  return cudaGetLastError() == cudaSuccess ? RL_OK : RL_ERR_CUDA;
}
