// lmhead.cu — rl_lmhead_logprobs: the LM-head projection fused with the
// log-softmax statistics, on the 5th-generation tensor cores (sm_103a).
//
// The logits the policy loss consumes are the actor's LM-head output
// (ainews.cool RL.cu article, section "技术深度解析": the actor network with
// its custom matrix multiplication).  For the log-probabilities of sampled
// tokens (the behaviour- and reference-policy log-probs of the update) only
// three numbers per row are needed, so this kernel never writes the
// R x V logits: it forms them tile by tile in tensor memory and folds each
// tile into online row statistics.
//
//   logits tile [128 rows x 256 vocab] = hidden[128 x D] . W[256 x D]^T
//
//   * warp 0 (one lane): TMA producer.  128B-swizzled tiles of hidden
//     (128 x 64) and W (256 x 64) through a 4-stage ring of 48 KB stages,
//     guarded by full/empty mbarriers.
//   * warp 1 (one lane): MMA issuer.  tcgen05.mma.kind::f16 (bf16 inputs,
//     fp32 accumulation), M=128 N=256 K=16, into one of two 256-column TMEM
//     accumulators; tcgen05.commit frees each smem stage and, after the last
//     K block, hands the accumulator to the epilogue.
//   * warps 2-5 (128 threads, one row each): tcgen05.ld of 32 columns at a
//     time, online (max, sum 2^x, sum 2^x x) per row, the sampled id's logit,
//     then lse, log-prob and entropy per row.  Freeing each accumulator lets
//     the MMAs of the next tile overlap this epilogue.
//   * Persistent over work units (128-row tile, vocabulary slice): the host
//     splits V into S slices so that the units spread evenly over the SMs
//     (S = 1 when the row tiles alone do).  Units are dealt out round-robin,
//     so the CTAs working at one time sweep the same slice of W in step and
//     share its tiles through L2.  With S > 1 each unit leaves per-row partial
//     statistics (max, sums, sampled logit) in the caller's workspace; the
//     last unit of a row tile to finish, found with a per-tile ticket, merges
//     the S partials in slice order (deterministic) and writes the outputs.
//   * Every mbarrier wait is bounded; on timeout the kernel raises an error
//     flag, waits for its own copies and tensor-core work, frees its tensor
//     memory and exits.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstring>
#include <mutex>

#include "tc_device.cuh"

namespace rl {
namespace {

constexpr int kBM = 128, kBN = 256, kBK = 64;   // tile shape (bf16: 64 elements = 128 B)
constexpr int kUmmaK = 16;                      // K of one tcgen05.mma.kind::f16
constexpr int kStagesL = 4;
constexpr uint32_t kStageA = kBM * kBK * 2;     // 16 KB
constexpr uint32_t kStageB = kBN * kBK * 2;     // 32 KB
constexpr int kThreadsL = 192;                  // producer, MMA, 4 epilogue warps
constexpr uint32_t kTmemCols = 2 * kBN;         // two fp32 accumulators
constexpr float kFloor = -1.0e30f;              // start of the running row maximum

struct LmSmem {
  alignas(1024) unsigned char a[kStagesL][kStageA];
  alignas(1024) unsigned char b[kStagesL][kStageB];
  unsigned long long full[kStagesL], empty[kStagesL];
  unsigned long long acc_full[2], acc_empty[2];
  unsigned long long drain;
  uint32_t tmem_base;
  int abort;
  int merge;  // this unit completes its row tile (vocabulary slices > 1)
};

struct LmArgs {
  long long R, D, V;
  uint32_t idesc;         // tcgen05 instruction descriptor (operand format)
  int n_mt, n_nt, n_slices;
  int group;              // row tiles per unit group
  unsigned int* tickets;  // [n_mt] (n_slices > 1)
  float4* partials;       // [n_slices][R]: (max, sum 2^x, sum 2^x x, sampled logit)
  const long long* ids;
  float* logp_out;
  float* entropy_out;
  float* lse_out;
  float4* row_partials;  // nullable: each row's (max, sum 2^x, sum 2^x x, sampled logit)
  unsigned int* status;  // nullable: RL_DEVERR_* bits
};

// First vocabulary tile of slice vs when n_nt tiles are cut into n_sl slices.
__device__ __forceinline__ int slice_begin(int vs, int n_nt, int n_sl) {
  return static_cast<int>(static_cast<long long>(vs) * n_nt / n_sl);
}

// Row tile and vocabulary slice of work unit u.  Units come in groups of g
// row tiles; inside a group they run slice by slice, so the CTAs working at
// one time share a slice of W and touch at most g hidden tiles (the host
// sizes g so that those tiles stay in L2).
__device__ __forceinline__ void unit_coords(int u, int n_mt, int n_sl, int g, int& mt, int& vs) {
  const int per_group = g * n_sl;
  const int grp = u / per_group;
  const int base = grp * g;
  const int gc = min(g, n_mt - base);
  const int within = u - grp * per_group;
  vs = within / gc;
  mt = base + within % gc;
}

// Instruction descriptor: fp32 D, A and B both bf16 or both fp16, both K-major.
__host__ __device__ constexpr uint32_t make_idesc(bool bf16) { return make_idesc_f16(bf16, kBM, kBN, false, false); }

template <bool kDrain>
__device__ __forceinline__ bool lm_wait(uint32_t bar, uint32_t parity, volatile int* abort) {
  return tc_wait<kDrain>(bar, parity, abort);
}

// ------------------------------------------------------------------ the kernel
__global__ void __launch_bounds__(kThreadsL, 1)
lmhead_logprobs_kernel(const __grid_constant__ CUtensorMap tmap_h, const __grid_constant__ CUtensorMap tmap_w,
                       const LmArgs a) {
  extern __shared__ unsigned char smem_raw[];
  // the swizzled tiles need 1024-byte alignment
  LmSmem& sm = *reinterpret_cast<LmSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  volatile int* abort_flag = &sm.abort;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n_mt = a.n_mt, n_nt = a.n_nt, n_sl = a.n_slices, n_units = n_mt * n_sl;
  const int n_kb = static_cast<int>((a.D + kBK - 1) / kBK);  // columns past D read as zeros

  if (tid == 0) {
    for (int s = 0; s < kStagesL; ++s) {
      mbar_init(smem_addr(&sm.full[s]), 1);
      mbar_init(smem_addr(&sm.empty[s]), 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(smem_addr(&sm.acc_full[s]), 1);
      mbar_init(smem_addr(&sm.acc_empty[s]), kBM);
    }
    mbar_init(smem_addr(&sm.drain), 1);
    sm.abort = 0;
    fence_mbar_init();
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap_h)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap_w)) : "memory");
  }
  if (warp == 1) {
    tmem_alloc(smem_addr(&sm.tmem_base), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;

  if (warp == 0) {
    // ---------------------------------------------------------------- TMA producer
    if (lane == 0) {
      uint32_t it = 0;
      bool stop = false;
      for (int u = blockIdx.x; u < n_units && !stop; u += gridDim.x) {
        int mt, vs;
        unit_coords(u, n_mt, n_sl, a.group, mt, vs);
        for (int nt = slice_begin(vs, n_nt, n_sl); nt < slice_begin(vs + 1, n_nt, n_sl) && !stop; ++nt) {
          for (int kb = 0; kb < n_kb; ++kb, ++it) {
            const uint32_t s = it % kStagesL, round = it / kStagesL;
            if (round > 0 && !lm_wait<false>(smem_addr(&sm.empty[s]), (round - 1) & 1, abort_flag)) {
              stop = true;
              break;
            }
            const uint32_t fb = smem_addr(&sm.full[s]);
            mbar_arrive_expect_tx(fb, kStageA + kStageB);
            tma_load_2d(smem_addr(sm.a[s]), &tmap_h, kb * kBK, mt * kBM, fb);
            tma_load_2d(smem_addr(sm.b[s]), &tmap_w, kb * kBK, nt * kBN, fb);
          }
        }
      }
      if (stop)  // copies already issued land before the CTA can exit
        for (uint32_t k = it > kStagesL ? it - kStagesL : 0; k < it; ++k)
          lm_wait<true>(smem_addr(&sm.full[k % kStagesL]), (k / kStagesL) & 1, abort_flag);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      uint32_t it = 0, acc_it = 0;
      bool stop = false, issued = false;
      for (int u = blockIdx.x; u < n_units && !stop; u += gridDim.x) {
        int mt, vs;
        unit_coords(u, n_mt, n_sl, a.group, mt, vs);
        for (int nt = slice_begin(vs, n_nt, n_sl); nt < slice_begin(vs + 1, n_nt, n_sl) && !stop; ++nt, ++acc_it) {
          const uint32_t buf = acc_it & 1, use = acc_it >> 1;
          if (use > 0 && !lm_wait<false>(smem_addr(&sm.acc_empty[buf]), (use - 1) & 1, abort_flag)) {
            stop = true;
            break;
          }
          tc_fence_after();
          const uint32_t d_tmem = tmem + buf * kBN;
          for (int kb = 0; kb < n_kb; ++kb, ++it) {
            const uint32_t s = it % kStagesL;
            if (!lm_wait<false>(smem_addr(&sm.full[s]), (it / kStagesL) & 1, abort_flag)) {
              stop = true;
              break;
            }
            tc_fence_after();
            const uint32_t a_base = smem_addr(sm.a[s]), b_base = smem_addr(sm.b[s]);
#pragma unroll
            for (int k = 0; k < kBK / kUmmaK; ++k)
              umma_f16(d_tmem, smem_desc_sw128(a_base + k * kUmmaK * 2), smem_desc_sw128(b_base + k * kUmmaK * 2),
                        a.idesc, (kb | k) != 0);
            issued = true;
            umma_commit(smem_addr(&sm.empty[s]));  // the stage is free once these MMAs have read it
          }
          if (stop) break;
          umma_commit(smem_addr(&sm.acc_full[buf]));  // accumulator ready for the epilogue
        }
      }
      if (stop && issued) {  // every MMA already issued completes before the memory is freed
        umma_commit(smem_addr(&sm.drain));
        lm_wait<true>(smem_addr(&sm.drain), 0, abort_flag);
      }
    }
  } else {
    // ---------------------------------------------------------------- epilogue
    const int q = warp & 3;          // TMEM lane quarter this warp may access
    const int r_in_tile = q * 32 + lane;
    const uint32_t lane_addr = static_cast<uint32_t>(q * 32) << 16;
    uint32_t acc_it = 0;
    bool stop = false;
    for (int u = blockIdx.x; u < n_units && !stop; u += gridDim.x) {
      int mt, vs;
      unit_coords(u, n_mt, n_sl, a.group, mt, vs);
      const long long row = static_cast<long long>(mt) * kBM + r_in_tile;
      const long long y = row < a.R ? a.ids[row] : -1;
      float m = kFloor, zy = -INFINITY;
      float2 s2 = make_float2(0.f, 0.f), t2 = make_float2(0.f, 0.f);
      for (int nt = slice_begin(vs, n_nt, n_sl); nt < slice_begin(vs + 1, n_nt, n_sl); ++nt, ++acc_it) {
        const uint32_t buf = acc_it & 1, use = acc_it >> 1;
        // warp-uniform outcome: the tensor-memory loads below are warp-collective
        if (!__all_sync(0xffffffffu, lm_wait<false>(smem_addr(&sm.acc_full[buf]), use & 1, abort_flag))) {
          stop = true;
          break;
        }
        tc_fence_after();
        const long long n0 = static_cast<long long>(nt) * kBN;
#pragma unroll 1
        for (int c = 0; c < kBN / 32; ++c) {
          float v[32];
          __syncwarp();
          tmem_ld32(tmem + lane_addr + buf * kBN + c * 32, v);
          const long long col0 = n0 + c * 32;
          const int nv = static_cast<int>(min(32LL, max(0LL, a.V - col0)));
          if (y >= col0 && y < col0 + 32) zy = select32(v, static_cast<int>(y - col0));
          float vm = kFloor;
#pragma unroll
          for (int i = 0; i < 32; ++i)
            if (i < nv) vm = max_nan(vm, v[i]);
          if (vm > m) {  // rescale the running sums to the new max
            const float d = (vm - m) * kLog2e;
            const float f = ex2_approx(-d);
            const float2 f2 = make_float2(f, f), nd2 = make_float2(-d, -d);
            t2 = __fmul2_rn(f2, __ffma2_rn(nd2, s2, t2));
            s2 = __fmul2_rn(f2, s2);
            m = vm;
          }
          const float2 L2 = make_float2(kLog2e, kLog2e);
          const float2 nmL = make_float2(-m * kLog2e, -m * kLog2e);
          if (nv == 32) {
#pragma unroll
            for (int i = 0; i < 32; i += 2) {
              const float2 x = __ffma2_rn(make_float2(v[i], v[i + 1]), L2, nmL);
              const float2 e = make_float2(ex2_approx(x.x), ex2_approx(x.y));
              s2 = __fadd2_rn(s2, e);
              t2 = __ffma2_rn(e, x, t2);
            }
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              if (i < nv) {
                const float x = fmaf(v[i], kLog2e, -m * kLog2e);
                const float e = ex2_approx(x);
                s2.x += e;
                t2.x = fmaf(e, x, t2.x);
              }
            }
          }
        }
        tc_fence_before();
        mbar_arrive(smem_addr(&sm.acc_empty[buf]));  // the MMA warp may overwrite this accumulator
      }
      float S = s2.x + s2.y, Tt = t2.x + t2.y;
      bool finish = true;
      if (n_sl > 1) {
        // Leave this slice's partial, then take the row tile's ticket.  Every
        // epilogue thread reaches these barriers once per unit, stopped or not.
        if (!stop && row < a.R)
          __stcg(&a.partials[static_cast<long long>(vs) * a.R + row], make_float4(m, S, Tt, zy));
        __threadfence();
        stop = named_barrier_or(1, 4 * 32, stop);
        if (tid == 2 * 32 && !stop)
          sm.merge = atomicInc(&a.tickets[mt], n_sl - 1) == static_cast<unsigned>(n_sl - 1);
        named_barrier(1, 4 * 32);
        finish = !stop && sm.merge;
        if (finish && row < a.R) {
          __threadfence();
          m = kFloor;
          for (int k = 0; k < n_sl; ++k)
            m = max_nan(m, __ldcg(&a.partials[static_cast<long long>(k) * a.R + row]).x);
          S = 0.f;
          Tt = 0.f;
          zy = -INFINITY;
          for (int k = 0; k < n_sl; ++k) {  // slice order: the result does not depend on arrival order
            const float4 pk = __ldcg(&a.partials[static_cast<long long>(k) * a.R + row]);
            const float d = (m - pk.x) * kLog2e;
            const float f = ex2_approx(-d);
            Tt += f * (pk.z - d * pk.y);
            S += f * pk.y;
            zy = fmaxf(zy, pk.w);
          }
        }
      }
      if (finish && !stop && row < a.R) {
        const float log2S = log2f(S);
        const float lse = fmaf(log2S, kLn2, m);
        const float H = kLn2 * (log2S - Tt / S);
        const bool y_ok = y >= 0 && y < a.V;
        if (a.logp_out) a.logp_out[row] = y_ok ? zy - lse : __int_as_float(0x7fc00000);
        if (a.entropy_out) a.entropy_out[row] = H;
        if (a.lse_out) a.lse_out[row] = lse;
        if (a.row_partials) a.row_partials[row] = make_float4(m, S, Tt, zy);
        if (!y_ok && a.status) atomicOr(a.status, RL_DEVERR_ID_RANGE);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (*abort_flag && tid == 0 && a.status) atomicOr(a.status, RL_DEVERR_TIMEOUT);
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ------------------------------------------------------------------ host side
std::mutex g_lm_mu;
int g_lm_attr_dev = -1;

rl_status encode_fn(EncodeTiled* out) { return tc_encode_fn(out); }

// 2-D tensor map [rows, cols] (row stride ld elements), box box_rows x 64, 128B swizzle.
bool make_map(EncodeTiled enc, CUtensorMap* map, CUtensorMapDataType dt, const void* base, long long rows,
              long long cols, long long ld, uint32_t box_rows) {
  return tc_make_map(enc, map, dt, base, rows, cols, ld, kBK, box_rows);
}

// Work split: S vocabulary slices per 128-row tile, chosen to minimise the
// busiest CTA's tile count under the round-robin deal (with half a tile of
// overhead per unit), within the workspace the caller gave.
constexpr int kMaxSlices = 1024;

struct LmPlan {
  int n_mt, n_nt, n_slices, grid, group;
  size_t ws_bytes;
};

// Hidden tiles the CTAs working at one time may touch: about 40 MB of L2,
// a third of it, leaving the rest to the weight slice being swept.
constexpr long long kHiddenL2Budget = 40LL << 20;

size_t ticket_bytes(long long n_mt) { return (static_cast<size_t>(n_mt) * 4 + 255) & ~size_t(255); }

size_t lm_ws_bytes(long long R, long long n_mt, int n_sl) {
  if (n_sl <= 1) return 0;
  return ticket_bytes(n_mt) + static_cast<size_t>(n_sl) * static_cast<size_t>(R) * 16;
}

LmPlan lm_plan(long long R, long long V, long long D, int sms, size_t ws_cap) {
  LmPlan p;
  p.n_mt = static_cast<int>((R + kBM - 1) / kBM);
  p.n_nt = static_cast<int>((V + kBN - 1) / kBN);
  auto cost = [&](int S) {
    const long long units = static_cast<long long>(p.n_mt) * S;
    const long long g = units < sms ? units : sms;
    return static_cast<double>((units + g - 1) / g) * ((p.n_nt + S - 1) / S + 0.5);
  };
  int best = 1;
  double best_cost = cost(1);
  const int s_max = p.n_nt < kMaxSlices ? p.n_nt : kMaxSlices;
  for (int S = 2; S <= s_max; ++S) {
    if (lm_ws_bytes(R, p.n_mt, S) > ws_cap || static_cast<long long>(p.n_mt) * S > (1LL << 30)) break;
    const double c = cost(S);
    if (c < best_cost * 0.999) {
      best = S;
      best_cost = c;
    }
  }
  p.n_slices = best;
  const long long units = static_cast<long long>(p.n_mt) * best;
  p.grid = static_cast<int>(units < sms ? units : sms);
  p.ws_bytes = lm_ws_bytes(R, p.n_mt, best);
  const long long tile_bytes = static_cast<long long>(kBM) * ((D + kBK - 1) / kBK) * kBK * 2;
  const long long g = kHiddenL2Budget / tile_bytes;
  p.group = static_cast<int>(g < 1 ? 1 : (g > p.n_mt ? p.n_mt : g));
  return p;
}

rl_status device_sms(int* sms) { return tc_device_sms(sms); }

bool lm_shape_ok(long long R, long long V) { return R >= 0 && R < (1LL << 31) && V >= 1 && V <= (1LL << 31); }

}  // namespace
}  // namespace rl

extern "C" size_t rl_lmhead_workspace_size(long long R, long long V) {
  using namespace rl;
  int sms = 0;
  if (R < 1 || !lm_shape_ok(R, V) || device_sms(&sms) != RL_OK) return 0;
  return lm_plan(R, V, 1024, sms, ~size_t(0)).ws_bytes;
}

extern "C" rl_status rl_lmhead_plan(long long R, long long D, long long V, size_t workspace_bytes, int sm_count,
                                    int* n_slices, int* grid, int* group, size_t* workspace_needed) {
  using namespace rl;
  if (R < 1 || !lm_shape_ok(R, V) || D < 8 || D % 8 != 0) return RL_ERR_SHAPE;
  int sms = sm_count;
  if (sms < 1 && device_sms(&sms) != RL_OK) return RL_ERR_CUDA;
  const LmPlan p = lm_plan(R, V, D, sms, workspace_bytes);
  if (n_slices) *n_slices = p.n_slices;
  if (grid) *grid = p.grid;
  if (group) *group = p.group;
  if (workspace_needed) *workspace_needed = p.ws_bytes;
  return RL_OK;
}

namespace {
rl_status lmhead_launch(const void* hidden, long long ld_h, const void* weight, long long ld_w, rl_dtype dtype,
                        long long R, long long D, long long V, const long long* ids, float* logp_out,
                        float* entropy_out, float* lse_out, float4* row_partials, unsigned int* status_dev,
                        void* workspace, size_t workspace_bytes, void* stream) {
  using namespace rl;
  if (dtype != RL_BF16 && dtype != RL_F16) return RL_ERR_DTYPE;
  if (!lm_shape_ok(R, V) || D < 8 || D % 8 != 0 || ld_h < D || ld_w < D) return RL_ERR_SHAPE;
  if (R == 0) return RL_OK;
  if (!hidden || !weight || !ids) return RL_ERR_NULL;
  if ((reinterpret_cast<uintptr_t>(hidden) & 15) || (reinterpret_cast<uintptr_t>(weight) & 15) ||
      ((ld_h * 2) & 15) || ((ld_w * 2) & 15) || (reinterpret_cast<uintptr_t>(workspace) & 15))
    return RL_ERR_ALIGN;
  EncodeTiled enc = nullptr;
  if (encode_fn(&enc) != RL_OK) return RL_ERR_CUDA;
  CUtensorMap mh, mw;
  const CUtensorMapDataType tdt =
      dtype == RL_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  if (!make_map(enc, &mh, tdt, hidden, R, D, ld_h, kBM) || !make_map(enc, &mw, tdt, weight, V, D, ld_w, kBN))
    return RL_ERR_CUDA;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || device_sms(&sms) != RL_OK) return RL_ERR_CUDA;
  const int smem = static_cast<int>(sizeof(LmSmem)) + 1024;
  {
    std::lock_guard<std::mutex> lock(g_lm_mu);
    if (g_lm_attr_dev != dev) {
      if (cudaFuncSetAttribute(lmhead_logprobs_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
          cudaSuccess)
        return RL_ERR_CUDA;
      g_lm_attr_dev = dev;
    }
  }
  const LmPlan plan = lm_plan(R, V, D, sms, workspace ? workspace_bytes : 0);
  LmArgs args;
  args.R = R;
  args.D = D;
  args.V = V;
  args.idesc = make_idesc(dtype == RL_BF16);
  args.n_mt = plan.n_mt;
  args.n_nt = plan.n_nt;
  args.n_slices = plan.n_slices;
  args.group = plan.group;
  args.tickets = plan.n_slices > 1 ? static_cast<unsigned int*>(workspace) : nullptr;
  args.partials = plan.n_slices > 1
                      ? reinterpret_cast<float4*>(static_cast<char*>(workspace) + ticket_bytes(plan.n_mt))
                      : nullptr;
  args.ids = ids;
  args.logp_out = logp_out;
  args.entropy_out = entropy_out;
  args.lse_out = lse_out;
  args.row_partials = row_partials;
  args.status = status_dev;
  lmhead_logprobs_kernel<<<plan.grid, kThreadsL, smem, static_cast<cudaStream_t>(stream)>>>(mh, mw, args);
  return cudaGetLastError() == cudaSuccess ? RL_OK : RL_ERR_CUDA;
}
}  // namespace

extern "C" rl_status rl_lmhead_logprobs(const void* hidden, long long ld_h, const void* weight, long long ld_w,
                                        rl_dtype dtype, long long R, long long D, long long V,
                                        const long long* ids,
                                        float* logp_out, float* entropy_out, float* lse_out,
                                        unsigned int* status_dev, void* workspace, size_t workspace_bytes,
                                        void* stream) {
  return lmhead_launch(hidden, ld_h, weight, ld_w, dtype, R, D, V, ids, logp_out, entropy_out, lse_out, nullptr,
                       status_dev, workspace, workspace_bytes, stream);
}

extern "C" rl_status rl_lmhead_row_partials(const void* hidden, long long ld_h, const void* weight,
                                            long long ld_w, rl_dtype dtype, long long R, long long D,
                                            long long V, const long long* ids, float* partials_out,
                                            unsigned int* status_dev, void* workspace,
                                            size_t workspace_bytes, void* stream) {
  if (R > 0 && !partials_out) return RL_ERR_NULL;
  if (reinterpret_cast<uintptr_t>(partials_out) & 15) return RL_ERR_ALIGN;
  return lmhead_launch(hidden, ld_h, weight, ld_w, dtype, R, D, V, ids, nullptr, nullptr, nullptr,
                       reinterpret_cast<float4*>(partials_out), status_dev, workspace, workspace_bytes, stream);
}
