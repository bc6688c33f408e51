// lmhead_grad.cu — the policy loss's gradient through the LM head on the
// 5th-generation tensor cores (sm_103a), without the logits in HBM.
//
// The actor's logits are its LM-head output z = hidden . W^T, computed by the
// pages' own matrix-multiplication kernels with 16-bit inputs and fp32
// accumulation (ainews.cool RL.cu article, section "技术深度解析", bullet
// 策略网络与价值网络 / policy and value networks; pitchhut.com RL.cu listing,
// "Key Features" item 1).  The loss gradient flows back through that
// product in three tensor-core GEMMs, each one template instantiation of the
// kernel below:
//
//   dlogits  dz = f(hidden . W^T)  [R x V]  A = hidden (K-major), B = W (K-major);
//            the logits tile is recomputed in tensor memory and the epilogue
//            turns it into the loss gradient with each row's coefficients
//            (the same arithmetic as the fused loss kernel's second pass),
//            so the logits themselves are never written;
//   dhidden  dH = dz . W           [R x D]  A = dz (K-major), B = W (N-major);
//   dweight  dW (+)= dz^T . hidden [V x D]  A = dz (M-major), B = hidden (N-major),
//            fp32 output, optionally added to what it holds.
//
//   * Tiles 128 x 256 x 64 (16-bit operands, 128-byte TMA swizzle), a 4-stage
//     ring of 48 KB stages, two 256-column fp32 accumulators in tensor memory
//     (the same structure as the forward LM-head kernel).
//   * warp 0 (one lane): TMA producer.  A K-major operand tile is one 2-D box
//     of 64 K-elements x rows; an M/N-major one is 64 K-rows x 64 elements
//     per box, 2 (A) or 4 (B) boxes side by side.
//   * warp 1 (one lane): MMA issuer (tcgen05.mma.kind::f16, M=128 N=256 K=16;
//     the instruction descriptor marks M/N-major operands as transposed).
//   * warps 2-5: epilogue, one accumulator row per thread.  dlogits stages
//     each warp's 32 rows x 64 columns in shared memory (128-byte swizzle, two
//     blocks per warp) and writes them with one TMA store; dhidden and dweight
//     store 16-bit or fp32 rows directly.
//   * Persistent over units of one tile each (the kernel also takes units of
//     several column tiles, n_sl < n_nt; for dlogits that measured slower).
//     dlogits units run in groups of row tiles that sweep W together (shared
//     through L2); the dhidden / dweight units put the column tiles of one
//     row tile next to each other, so the CTAs working at one time read the
//     same dz tiles.
//   * Every mbarrier wait is bounded; on timeout the kernel raises an error
//     flag, waits for its own copies and tensor-core work, frees its tensor
//     memory and exits.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cmath>
#include <cstring>
#include <mutex>

#include "tc_device.cuh"

namespace rl {
namespace {

constexpr int kGM = 128, kGN = 256, kGK = 64;
constexpr int kGStages = 4;
constexpr uint32_t kGStageA = kGM * kGK * 2;  // 16 KB
constexpr uint32_t kGStageB = kGN * kGK * 2;  // 32 KB
constexpr uint32_t kMnBlock = kGK * 128;      // one 64-element M/N block of an M/N-major tile: 64 K-rows x 128 B
// Epilogue shape (compile-time knobs; the defaults are the shipped configuration):
// RLG_EPI_WARPS epilogue warps (4: one warpgroup; 8: two, each on half of a
// tile's columns), RLG_STAGE_BUFS staging blocks per warp for dlogits, and
// RLG_STORE how dlogits leaves the staging block: 0 a TMA store, 1 the same
// with an evict-first L2 hint, 2 coalesced 16-byte stores by the warp.
#ifndef RLG_EPI_WARPS
#define RLG_EPI_WARPS 4
#endif
#ifndef RLG_STAGE_BUFS
#define RLG_STAGE_BUFS 2
#endif
#ifndef RLG_STORE
#define RLG_STORE 0
#endif
// RLG_CLUSTER CTAs per cluster (1 or 2).  With 2, the CTAs of a pair take
// row tiles 2p and 2p + 1 of the same column tile: each TMA-loads half of the
// B tile and multicasts it to both, so each CTA reads 32 KB per K block from
// L2 instead of 48 KB, and each MMA commit frees the stage in both CTAs.
#ifndef RLG_CLUSTER
#define RLG_CLUSTER 1
#endif
constexpr int kCl = RLG_CLUSTER;
static_assert(kCl == 1 || kCl == 2, "one CTA or a pair per cluster");
constexpr int kEpiWarps = RLG_EPI_WARPS;
constexpr int kEpiGroups = kEpiWarps / 4;          // warpgroups, each on kGN / kEpiGroups columns
constexpr int kStageBufs = RLG_STAGE_BUFS;
constexpr int kGThreads = 64 + 32 * kEpiWarps;     // producer, MMA, epilogue warps
static_assert(kEpiWarps == 4 || kEpiWarps == 8, "one or two epilogue warpgroups");
constexpr uint32_t kGTmemCols = 2 * kGN;      // two fp32 accumulators
constexpr long long kHiddenL2Bytes = 40LL << 20;  // row tiles a dlogits unit group may keep in L2

enum GemmEpi { kEpiDlogits = 0, kEpiStore16 = 1, kEpiAccF32 = 2 };

constexpr uint32_t kStageRows = 32, kStageBytes = kStageRows * 128;  // one warp's 32 rows x 64 columns

struct GSmem {
  alignas(1024) unsigned char a[kGStages][kGStageA];
  alignas(1024) unsigned char b[kGStages][kGStageB];
  // dlogits: each epilogue warp stages 32 rows x 64 columns of dz here (128-byte
  // swizzled rows) for a TMA store
  alignas(1024) unsigned char stage[kEpiWarps][kStageBufs][kStageBytes];
  unsigned long long full[kGStages], empty[kGStages];
  unsigned long long acc_full[2], acc_empty[2];
  unsigned long long drain;
  uint32_t tmem_base;
  int abort;
};

static_assert(sizeof(GSmem) + 1024 <= 232448, "ring, staging and barriers fit the 227 KB a CTA may use");

struct GArgs {
  long long M, N;
  uint32_t idesc;
  int n_mt, n_nt, n_kb, group;
  int n_sl;              // column slices: a unit is (row tile, slice of n_nt / n_sl column tiles)
  void* out;             // row-major [M, ld_out]: 16-bit (dlogits, dhidden) or fp32 (dweight)
  long long ld_out;
  int out_f16;           // 16-bit outputs: fp16 instead of bf16
  int accumulate;        // fp32 output: add to what it holds
  const float4* coef;    // dlogits: per row (cL, a0, a1, gy)
  const long long* ids;  // dlogits: sampled id per row
  unsigned int* status;  // nullable: RL_DEVERR_* bits
};

// Pack 32 floats to 16-bit pairs (round to nearest even) and store 64 bytes.
__device__ __forceinline__ void store16x32(unsigned char* p, const float (&v)[32], bool f16) {
  uint32_t u[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    if (f16) {
      __half2 h = __floats2half2_rn(v[2 * i], v[2 * i + 1]);
      u[i] = *reinterpret_cast<uint32_t*>(&h);
    } else {
      __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
      u[i] = *reinterpret_cast<uint32_t*>(&h);
    }
  }
  uint4* q = reinterpret_cast<uint4*>(p);
#pragma unroll
  for (int i = 0; i < 4; ++i) q[i] = make_uint4(u[4 * i], u[4 * i + 1], u[4 * i + 2], u[4 * i + 3]);
}

__device__ __forceinline__ void store16(unsigned char* p, float v, bool f16) {
  if (f16)
    *reinterpret_cast<__half*>(p) = __float2half_rn(v);
  else
    *reinterpret_cast<__nv_bfloat16*>(p) = __float2bfloat16_rn(v);
}

// 2^x (a0 + a1 x) with x = z_v log2(e) - cL for one row's 32 logits: the
// loss gradient without the sampled id's -gy term.
__device__ __forceinline__ void dlogits32(float (&v)[32], float cL, float a0, float a1, bool p_term) {
  const float2 L2 = make_float2(kLog2e, kLog2e);
  const float2 ncL = make_float2(-cL, -cL);
  const float2 A0 = make_float2(a0, a0), A1 = make_float2(a1, a1);
#pragma unroll
  for (int i = 0; i < 32; i += 2) {
    const float2 x = __ffma2_rn(make_float2(v[i], v[i + 1]), L2, ncL);
    const float2 p = make_float2(ex2_approx(x.x), ex2_approx(x.y));
    const float2 r = __fmul2_rn(p, __ffma2_rn(A1, x, A0));
    v[i] = p_term ? r.x : 0.f;
    v[i + 1] = p_term ? r.y : 0.f;
  }
}

__device__ __forceinline__ uint32_t pack16x2(float lo, float hi, bool f16) {
  if (f16) {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
  }
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}
__device__ __forceinline__ void st_shared_u16(uint32_t addr, uint16_t v) {
  asm volatile("st.shared.b16 [%0], %1;" ::"r"(addr), "h"(v) : "memory");
}

// ------------------------------------------------------------------ the kernel
template <bool kAMN, bool kBMN, int kEpi>
__global__ void __launch_bounds__(kGThreads, 1)
lmhead_grad_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                   const __grid_constant__ CUtensorMap tmap_out, const GArgs a) {
  extern __shared__ unsigned char smem_raw[];
  GSmem& sm = *reinterpret_cast<GSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  volatile int* abort_flag = &sm.abort;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // units are (row tile, or pair of row tiles with clusters of two CTAs;
  // slice of column tiles), the slice's tiles taken in order
  const int n_nt = a.n_nt, n_kb = a.n_kb, n_sl = a.n_sl;
  const int n_mt = (a.n_mt + kCl - 1) / kCl, n_units = n_mt * n_sl;
  const uint32_t crank = kCl > 1 ? cluster_rank() : 0;
  const int cid = kCl > 1 ? static_cast<int>(cluster_id()) : static_cast<int>(blockIdx.x);
  const int ncl = kCl > 1 ? static_cast<int>(cluster_count()) : static_cast<int>(gridDim.x);
  constexpr uint16_t kMask = static_cast<uint16_t>((1u << kCl) - 1);

  if (tid == 0) {
    for (int s = 0; s < kGStages; ++s) {
      mbar_init(smem_addr(&sm.full[s]), 1);
      mbar_init(smem_addr(&sm.empty[s]), kCl);  // freed by the MMA commits of every CTA that writes it
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(smem_addr(&sm.acc_full[s]), 1);
      mbar_init(smem_addr(&sm.acc_empty[s]), 32 * kEpiWarps);
    }
    mbar_init(smem_addr(&sm.drain), 1);
    sm.abort = 0;
    fence_mbar_init();
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap_a)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap_b)) : "memory");
    if (kEpi == kEpiDlogits)
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap_out)) : "memory");
  }
  if (warp == 1) {
    tmem_alloc(smem_addr(&sm.tmem_base), kGTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  if (kCl > 1) cluster_sync_all();  // the peer's barriers exist before any multicast reaches them
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;

  if (warp == 0) {
    // ---------------------------------------------------------------- TMA producer
    if (lane == 0) {
      uint32_t it = 0;
      bool stop = false;
      for (int u = cid; u < n_units && !stop; u += ncl) {
        int mt, vs;
        unit_tile(u, n_mt, n_sl, a.group, mt, vs);
        mt = mt * kCl + static_cast<int>(crank);
        for (int nt = slice_first(vs, n_nt, n_sl); nt < slice_first(vs + 1, n_nt, n_sl) && !stop; ++nt)
        for (int kb = 0; kb < n_kb; ++kb, ++it) {
          const uint32_t s = it % kGStages, round = it / kGStages;
          if (round > 0 && !tc_wait<false>(smem_addr(&sm.empty[s]), (round - 1) & 1, abort_flag)) {
            stop = true;
            break;
          }
          const uint32_t fb = smem_addr(&sm.full[s]);
          mbar_arrive_expect_tx(fb, kGStageA + kGStageB);
          if (kAMN) {
#pragma unroll
            for (int j = 0; j < kGM / 64; ++j)
              tma_load_2d(smem_addr(sm.a[s]) + j * kMnBlock, &tmap_a, mt * kGM + j * 64, kb * kGK, fb);
          } else {
            tma_load_2d(smem_addr(sm.a[s]), &tmap_a, kb * kGK, mt * kGM, fb);
          }
          // this CTA's share of the B tile (all of it without a cluster)
          if (kBMN) {
#pragma unroll
            for (int j = 0; j < kGN / 64 / kCl; ++j) {
              const int jj = static_cast<int>(crank) * (kGN / 64 / kCl) + j;
              if (kCl > 1)
                tma_load_2d_mc(smem_addr(sm.b[s]) + jj * kMnBlock, &tmap_b, nt * kGN + jj * 64, kb * kGK, fb, kMask);
              else
                tma_load_2d(smem_addr(sm.b[s]) + jj * kMnBlock, &tmap_b, nt * kGN + jj * 64, kb * kGK, fb);
            }
          } else {
            const int r0 = static_cast<int>(crank) * (kGN / kCl);
            if (kCl > 1)
              tma_load_2d_mc(smem_addr(sm.b[s]) + r0 * 128, &tmap_b, kb * kGK, nt * kGN + r0, fb, kMask);
            else
              tma_load_2d(smem_addr(sm.b[s]), &tmap_b, kb * kGK, nt * kGN, fb);
          }
        }
      }
      if (stop)  // copies already issued land before the CTA can exit
        for (uint32_t k = it > kGStages ? it - kGStages : 0; k < it; ++k)
          tc_wait<true>(smem_addr(&sm.full[k % kGStages]), (k / kGStages) & 1, abort_flag);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      uint32_t it = 0, acc_it = 0;
      bool stop = false, issued = false;
      int mt_u = 0, vs = 0, nt = 0, nt_end = 0, u = cid - ncl;
      while (!stop) {
        if (nt == nt_end) {  // next unit: its slice's column tiles
          u += ncl;
          if (u >= n_units) break;
          unit_tile(u, n_mt, n_sl, a.group, mt_u, vs);
          nt = slice_first(vs, n_nt, n_sl);
          nt_end = slice_first(vs + 1, n_nt, n_sl);
          if (nt == nt_end) continue;
        }
        ++nt;
        const uint32_t buf = acc_it & 1, use = acc_it >> 1;
        ++acc_it;
        if (use > 0 && !tc_wait<false>(smem_addr(&sm.acc_empty[buf]), (use - 1) & 1, abort_flag)) {
          stop = true;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem + buf * kGN;
        for (int kb = 0; kb < n_kb; ++kb, ++it) {
          const uint32_t s = it % kGStages;
          if (!tc_wait<false>(smem_addr(&sm.full[s]), (it / kGStages) & 1, abort_flag)) {
            stop = true;
            break;
          }
          tc_fence_after();
          const uint32_t a_base = smem_addr(sm.a[s]), b_base = smem_addr(sm.b[s]);
#pragma unroll
          for (int k = 0; k < kGK / 16; ++k) {
            // K-major: the next 16 K are 32 bytes further along each row; M/N-major:
            // 16 rows (two 8-row atoms) further down each 64-element block.
            const uint64_t ad = kAMN ? smem_desc_sw128_mn(a_base + k * 16 * 128, kMnBlock)
                                     : smem_desc_sw128(a_base + k * 32);
            const uint64_t bd = kBMN ? smem_desc_sw128_mn(b_base + k * 16 * 128, kMnBlock)
                                     : smem_desc_sw128(b_base + k * 32);
            umma_f16(d_tmem, ad, bd, a.idesc, (kb | k) != 0);
          }
          issued = true;
          // the stage is free once these MMAs have read it (in every CTA that loads into it)
          if (kCl > 1)
            umma_commit_mc(smem_addr(&sm.empty[s]), kMask);
          else
            umma_commit(smem_addr(&sm.empty[s]));
        }
        if (stop) break;
        umma_commit(smem_addr(&sm.acc_full[buf]));  // accumulator ready for the epilogue
      }
      if (stop && issued) {  // every MMA already issued completes before the memory is freed
        umma_commit(smem_addr(&sm.drain));
        tc_wait<true>(smem_addr(&sm.drain), 0, abort_flag);
      }
    }
  } else {
    // ---------------------------------------------------------------- epilogue
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    const int half = (warp - 2) / 4;  // which part of the tile's columns this warp takes
    const int r_in_tile = q * 32 + lane;
    const uint32_t lane_addr = static_cast<uint32_t>(q * 32) << 16;
    const bool f16 = a.out_f16 != 0;
    uint32_t acc_it = 0, blk = 0;
#if RLG_STORE == 1
    const uint64_t store_pol = policy_evict_first();
#endif
    bool stop = false;
    for (int u = cid; u < n_units && !stop; u += ncl) {
      int mt, vs;
      unit_tile(u, n_mt, n_sl, a.group, mt, vs);
      mt = mt * kCl + static_cast<int>(crank);
      for (int nt = slice_first(vs, n_nt, n_sl); nt < slice_first(vs + 1, n_nt, n_sl); ++nt, ++acc_it) {
      const long long row = static_cast<long long>(mt) * kGM + r_in_tile;
      const bool row_ok = row < a.M;
      float cL = 0.f, a0 = 0.f, a1 = 0.f, gy = 0.f;
      long long y = -1;
      if (kEpi == kEpiDlogits && row_ok) {
        const float4 c = a.coef[row];
        cL = c.x;
        a0 = c.y;
        a1 = c.z;
        gy = c.w;
        y = a.ids[row];
      }
      const uint32_t buf = acc_it & 1, use = acc_it >> 1;
      // warp-uniform outcome: the tensor-memory loads below are warp-collective
      if (!__all_sync(0xffffffffu, tc_wait<false>(smem_addr(&sm.acc_full[buf]), use & 1, abort_flag))) {
        stop = true;
        break;
      }
      tc_fence_after();
      // a row with no probability term (a masked row, or g = c_ent = 0) keeps
      // only the -gy of its sampled id: 2^x is never formed for it (used only
      // now, so the coefficient loads above overlap the accumulator wait)
      const bool p_term = a0 != 0.f || a1 != 0.f;
      const long long n0 = static_cast<long long>(nt) * kGN;
      if (kEpi == kEpiDlogits) {
        // 64 columns at a time: two tensor-memory loads into this warp's staging
        // block (row = lane, 16-byte chunk c of a row at position c ^ (row % 8),
        // the TMA 128-byte swizzle), then one TMA store of the 32 x 64 box; the
        // store clips rows past R and columns past V.
#pragma unroll 1
        for (int c2 = half * (kGN / 64 / kEpiGroups); c2 < (half + 1) * (kGN / 64 / kEpiGroups); ++c2, ++blk) {
          const uint32_t stage = smem_addr(sm.stage[warp - 2][blk % kStageBufs]);
          const uint32_t sbuf = stage + lane * 128;
#if RLG_STORE != 2
          // the store that last read this staging block is done with it
          if (lane == 0) {
            if (kStageBufs == 1)
              bulk_wait_all_read();
            else
              bulk_wait_read_1();
          }
#endif
          __syncwarp();
          float v64[64];
          tmem_ld64(tmem + lane_addr + buf * kGN + c2 * 64, v64);
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            float v[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = v64[h * 32 + i];
            dlogits32(v, cL, a0, a1, p_term);
#pragma unroll
            for (int j = 0; j < 4; ++j)
              st_shared_v4(sbuf + (((h * 4 + j) ^ (lane & 7)) << 4), pack16x2(v[8 * j], v[8 * j + 1], f16),
                           pack16x2(v[8 * j + 2], v[8 * j + 3], f16), pack16x2(v[8 * j + 4], v[8 * j + 5], f16),
                           pack16x2(v[8 * j + 6], v[8 * j + 7], f16));
            const long long jy = y - (n0 + c2 * 64 + h * 32);
            const bool has_y = jy >= 0 && jy < 32;
            if (__any_sync(0xffffffffu, has_y) && has_y) {  // rare: the sampled id's column
              const int e = h * 32 + static_cast<int>(jy);
              const float dy = select32(v, static_cast<int>(jy)) - gy;
              const uint32_t bits = pack16x2(dy, 0.f, f16) & 0xffffu;
              st_shared_u16(sbuf + (((e >> 3) ^ (lane & 7)) << 4) + (e & 7) * 2, static_cast<uint16_t>(bits));
            }
          }
#if RLG_STORE == 2
          // each lane sends 16-byte pieces: four full 128-byte rows per instruction
          __syncwarp();
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int r = i * 4 + (lane >> 3), c = lane & 7;
            const uint4 w = ld_shared_v4(stage + r * 128 + ((c ^ (r & 7)) << 4));
            const long long grow = static_cast<long long>(mt) * kGM + q * 32 + r;
            const long long gcol = n0 + c2 * 64 + c * 8;
            if (grow < a.M && gcol < a.N) {
              unsigned char* o = static_cast<unsigned char*>(a.out) + (grow * a.ld_out + gcol) * 2;
              if (gcol + 8 <= a.N) {
                *reinterpret_cast<uint4*>(o) = w;
              } else {
                const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
                for (int e = 0; e < a.N - gcol; ++e)
                  *reinterpret_cast<uint16_t*>(o + 2 * e) = static_cast<uint16_t>(ww[e >> 1] >> (16 * (e & 1)));
              }
            }
          }
          __syncwarp();
#else
          fence_proxy_async_shared();  // this lane's staging writes, before the async proxy reads them
          __syncwarp();
          if (lane == 0) {
#if RLG_STORE == 1
            tma_store_2d_hint(&tmap_out, static_cast<int>(n0 + c2 * 64), mt * kGM + q * 32, stage, store_pol);
#else
            tma_store_2d(&tmap_out, static_cast<int>(n0 + c2 * 64), mt * kGM + q * 32, stage);
#endif
            bulk_commit();
          }
#endif
        }
      }
#pragma unroll 1
      for (int c = half * (kGN / 32 / kEpiGroups); kEpi != kEpiDlogits && c < (half + 1) * (kGN / 32 / kEpiGroups);
           ++c) {
        float v[32];
        __syncwarp();
        tmem_ld32(tmem + lane_addr + buf * kGN + c * 32, v);
        const long long col0 = n0 + c * 32;
        if (!row_ok || col0 >= a.N) continue;
        const int nv = static_cast<int>(min(32LL, a.N - col0));
        if (kEpi == kEpiAccF32) {
          float* o = static_cast<float*>(a.out) + row * a.ld_out + col0;
          if (nv == 32) {
            float4* o4 = reinterpret_cast<float4*>(o);
            if (a.accumulate) {
              float4 old[8];
#pragma unroll
              for (int i = 0; i < 8; ++i) old[i] = o4[i];
#pragma unroll
              for (int i = 0; i < 8; ++i)
                o4[i] = make_float4(old[i].x + v[4 * i], old[i].y + v[4 * i + 1], old[i].z + v[4 * i + 2],
                                    old[i].w + v[4 * i + 3]);
            } else {
#pragma unroll
              for (int i = 0; i < 8; ++i) o4[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
            }
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (i < nv) o[i] = a.accumulate ? o[i] + v[i] : v[i];
          }
        } else {
          unsigned char* o = static_cast<unsigned char*>(a.out) + (row * a.ld_out + col0) * 2;
          if (nv == 32) {
            store16x32(o, v, f16);
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (i < nv) store16(o + 2 * i, v[i], f16);
          }
        }
      }
      tc_fence_before();
      mbar_arrive(smem_addr(&sm.acc_empty[buf]));  // the MMA warp may overwrite this accumulator
      }
    }
    if (kEpi == kEpiDlogits && lane == 0) bulk_wait_all();  // every store done before the CTA exits
  }

  tc_fence_before();
  __syncthreads();
  if (*abort_flag && tid == 0 && a.status) atomicOr(a.status, RL_DEVERR_TIMEOUT);
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kGTmemCols);
  }
  if (kCl > 1) cluster_sync_all();  // no CTA leaves while its peer may still multicast into it
}

// ------------------------------------------------------------------ host side
template <bool kAMN, bool kBMN, int kEpi>
rl_status launch_grad(const CUtensorMap& ma, const CUtensorMap& mb, const CUtensorMap& mo, const GArgs& args,
                      cudaStream_t stream) {
  static std::mutex mu;
  static int attr_dev = -1;
  const int smem = static_cast<int>(sizeof(GSmem)) + 1024;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || tc_device_sms(&sms) != RL_OK) return RL_ERR_CUDA;
  static int max_clusters = 0;
  auto fn = lmhead_grad_kernel<kAMN, kBMN, kEpi>;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kCl;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(kGThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (attr_dev != dev) {
      if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
        return RL_ERR_CUDA;
      int n = sms;
      if (kCl > 1) {
        cfg.gridDim = dim3(kCl);
        if (cudaOccupancyMaxActiveClusters(&n, fn, &cfg) != cudaSuccess || n < 1) return RL_ERR_CUDA;
      }
      max_clusters = n;
      attr_dev = dev;
    }
  }
  const long long units = static_cast<long long>((args.n_mt + kCl - 1) / kCl) * args.n_sl;
  if (units == 0) return RL_OK;
  const long long n_clusters = units < max_clusters ? units : max_clusters;
  cfg.gridDim = dim3(static_cast<unsigned>(n_clusters * kCl));
  return cudaLaunchKernelEx(&cfg, fn, ma, mb, mo, args) == cudaSuccess ? RL_OK : RL_ERR_CUDA;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

// Shapes every entry point accepts: 16-bit formats, R < 2^31 rows, V < 2^31
// columns, D a positive multiple of 8, row strides of 16-byte multiples.
rl_status check_common(rl_dtype dtype, long long R, long long D, long long V) {
  if (dtype != RL_BF16 && dtype != RL_F16) return RL_ERR_DTYPE;
  if (R < 0 || R >= (1LL << 31) || V < 1 || V >= (1LL << 31) || D < 8 || D % 8 != 0 || D >= (1LL << 31))
    return RL_ERR_SHAPE;
  return RL_OK;
}

bool ld_ok(long long ld, long long cols) { return ld >= cols && (ld * 2) % 16 == 0; }

CUtensorMapDataType tmap_type(rl_dtype dtype) {
  return dtype == RL_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
}

GArgs base_args(long long M, long long N, long long K, bool bf16, bool a_mn, bool b_mn) {
  GArgs g;
  std::memset(&g, 0, sizeof(g));
  g.M = M;
  g.N = N;
  g.idesc = make_idesc_f16(bf16, kGM, kGN, a_mn, b_mn);
  g.n_mt = static_cast<int>((M + kGM - 1) / kGM);
  g.n_nt = static_cast<int>((N + kGN - 1) / kGN);
  g.n_kb = static_cast<int>((K + kGK - 1) / kGK);
  g.group = 1;
  g.n_sl = g.n_nt;  // one column tile per unit
  return g;
}

}  // namespace
}  // namespace rl

using namespace rl;

extern "C" rl_status rl_lmhead_dlogits(const void* hidden, long long ld_h, const void* weight, long long ld_w,
                                       rl_dtype dtype, long long R, long long D, long long V,
                                       const long long* ids, const float* row_coef, void* dlogits,
                                       long long ld_dz, unsigned int* status_dev, void* stream) {
  rl_status st = check_common(dtype, R, D, V);
  if (st != RL_OK) return st;
  if (!ld_ok(ld_h, D) || !ld_ok(ld_w, D) || !ld_ok(ld_dz, V)) return RL_ERR_SHAPE;
  if (R == 0) return RL_OK;
  if (!hidden || !weight || !ids || !row_coef || !dlogits) return RL_ERR_NULL;
  if (!aligned16(hidden) || !aligned16(weight) || !aligned16(row_coef) || !aligned16(dlogits)) return RL_ERR_ALIGN;
  EncodeTiled enc = nullptr;
  if (tc_encode_fn(&enc) != RL_OK) return RL_ERR_CUDA;
  CUtensorMap ma, mb, mo;
  if (!tc_make_map(enc, &ma, tmap_type(dtype), hidden, R, D, ld_h, kGK, kGM) ||
      !tc_make_map(enc, &mb, tmap_type(dtype), weight, V, D, ld_w, kGK, kGN / kCl) ||
      !tc_make_map(enc, &mo, tmap_type(dtype), dlogits, R, V, ld_dz, 64, kStageRows))
    return RL_ERR_CUDA;
  GArgs g = base_args(R, V, D, dtype == RL_BF16, false, false);
  const long long tile_bytes = static_cast<long long>(kGM) * g.n_kb * kGK * 2;
  const long long grp = kHiddenL2Bytes / tile_bytes / kCl;  // groups of row-tile pairs
  g.group = static_cast<int>(grp < 1 ? 1 : (grp > g.n_mt ? g.n_mt : grp));
  g.out = dlogits;
  g.ld_out = ld_dz;
  g.out_f16 = dtype == RL_F16;
  g.coef = reinterpret_cast<const float4*>(row_coef);
  g.ids = ids;
  g.status = status_dev;
  return launch_grad<false, false, kEpiDlogits>(ma, mb, mo, g, static_cast<cudaStream_t>(stream));
}

extern "C" rl_status rl_lmhead_dhidden(const void* dlogits, long long ld_dz, const void* weight, long long ld_w,
                                       rl_dtype dtype, long long R, long long D, long long V, void* dhidden,
                                       long long ld_dh, unsigned int* status_dev, void* stream) {
  rl_status st = check_common(dtype, R, D, V);
  if (st != RL_OK) return st;
  if (!ld_ok(ld_dz, V) || !ld_ok(ld_w, D) || !ld_ok(ld_dh, D)) return RL_ERR_SHAPE;
  if (R == 0) return RL_OK;
  if (!dlogits || !weight || !dhidden) return RL_ERR_NULL;
  if (!aligned16(dlogits) || !aligned16(weight) || !aligned16(dhidden)) return RL_ERR_ALIGN;
  EncodeTiled enc = nullptr;
  if (tc_encode_fn(&enc) != RL_OK) return RL_ERR_CUDA;
  CUtensorMap ma, mb;
  if (!tc_make_map(enc, &ma, tmap_type(dtype), dlogits, R, V, ld_dz, kGK, kGM) ||
      !tc_make_map(enc, &mb, tmap_type(dtype), weight, V, D, ld_w, 64, kGK))
    return RL_ERR_CUDA;
  GArgs g = base_args(R, D, V, dtype == RL_BF16, false, true);
  g.out = dhidden;
  g.ld_out = ld_dh;
  g.out_f16 = dtype == RL_F16;
  g.status = status_dev;
  return launch_grad<false, true, kEpiStore16>(ma, mb, mb, g, static_cast<cudaStream_t>(stream));
}

extern "C" rl_status rl_lmhead_dweight(const void* dlogits, long long ld_dz, const void* hidden, long long ld_h,
                                       rl_dtype dtype, long long R, long long D, long long V, float* dweight,
                                       long long ld_dw, int accumulate, unsigned int* status_dev,
                                       void* stream) {
  rl_status st = check_common(dtype, R, D, V);
  if (st != RL_OK) return st;
  if (!ld_ok(ld_dz, V) || !ld_ok(ld_h, D) || ld_dw < D || ld_dw % 4 != 0) return RL_ERR_SHAPE;
  if (!dweight) return RL_ERR_NULL;
  if (!aligned16(dweight)) return RL_ERR_ALIGN;
  if (R == 0) {
    // an empty batch contributes nothing: overwrite mode leaves a zero gradient
    if (!accumulate &&
        cudaMemset2DAsync(dweight, static_cast<size_t>(ld_dw) * 4, 0, static_cast<size_t>(D) * 4,
                          static_cast<size_t>(V), static_cast<cudaStream_t>(stream)) != cudaSuccess)
      return RL_ERR_CUDA;
    return RL_OK;
  }
  if (!dlogits || !hidden) return RL_ERR_NULL;
  if (!aligned16(dlogits) || !aligned16(hidden)) return RL_ERR_ALIGN;
  EncodeTiled enc = nullptr;
  if (tc_encode_fn(&enc) != RL_OK) return RL_ERR_CUDA;
  CUtensorMap ma, mb;
  if (!tc_make_map(enc, &ma, tmap_type(dtype), dlogits, R, V, ld_dz, 64, kGK) ||
      !tc_make_map(enc, &mb, tmap_type(dtype), hidden, R, D, ld_h, 64, kGK))
    return RL_ERR_CUDA;
  GArgs g = base_args(V, D, R, dtype == RL_BF16, true, true);
  g.out = dweight;
  g.ld_out = ld_dw;
  g.accumulate = accumulate != 0;
  g.status = status_dev;
  return launch_grad<true, true, kEpiAccF32>(ma, mb, mb, g, static_cast<cudaStream_t>(stream));
}
