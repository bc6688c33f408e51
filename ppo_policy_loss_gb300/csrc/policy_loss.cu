// policy_loss.cu — rl_policy_loss_fwd_bwd: the fused policy loss and its
// logits gradient in one launch (sm_103a).
//
// The RL.cu pages describe a single fused "PPO update kernel" (ainews.cool
// RL.cu article, section "技术深度解析", bullet "PPO 更新内核") that computes
// the whole loss, with the KL penalty and reward normalisation of the
// paragraph after its benchmark table, in one launch to avoid global-memory
// round trips.  This kernel is that step for GB300, designed around HBM:
//
//   * Persistent grid; CTA q takes rows q, q + Q, ...  Two builds of this
//     source (see RL_SHORT_ROWS below): one CTA per SM with 16 consumer
//     warps and 32 KB chunks for rows longer than 100 KB, two CTAs per SM
//     with 8 consumer warps and 16 KB chunks for shorter rows.  The figures
//     in the rest of this comment are the long-row build's.
//   * One producer warp streams the valid rows with 1-D bulk copies
//     (cp.async.bulk) into a ring of 6 x 32 KB shared-memory chunks guarded
//     by full/empty mbarriers, running ahead of the consumers by up to the
//     whole ring.  32 KB chunks give each consumer thread four 16-byte
//     vectors per chunk, independent work that hides latency.
//   * Two row modes:
//       - resident: a row that fits the ring twice over (at most 2 chunks)
//         is loaded once and kept in shared memory for both passes;
//       - streaming: a longer row (151936 bf16 logits = 10 chunks) is streamed
//         twice: the first load keeps its L2 lines (evict-last), the second
//         pass re-reads them from L2 (evict-first).  Logits still cross the
//         HBM bus once, and the ring is always free to prefetch.  When no
//         row is masked the second pass runs in reverse chunk order.
//   * Consumer warps: pass 1 keeps a per-thread online (max, sum 2^x,
//     sum 2^x * x) in packed fp32x2 with independent accumulator chains;
//     each warp then reduces its lanes and publishes one partial.  In the
//     short-row build a row's last, partly filled chunk is padded in shared
//     memory with the format's floor and taken by the same routine as a full
//     chunk (the row warp removes the padding's share in the rows where it
//     can have one); long rows keep a predicated routine for it.  Pass 2
//     writes the gradient with 16-byte streaming stores.  The entropy term
//     is a template argument, so each launch runs only the pass-2 code it
//     needs.
//   * A row warp merges the consumer warps' partials of each row and turns
//     them into the row's loss terms and pass-2 coefficients: a long chain
//     of dependent scalar arithmetic, run once per row instead of once per
//     consumer warp.  Two rows are in flight between the consumers and the
//     row warp.  When no row of the batch is masked the consumers run the
//     first chunks of the next row's pass 1 before a row's pass 2 (long
//     rows one chunk; short rows two, or the whole row if it has at most
//     four), which covers the row warp's time for that row.  Long rows pass
//     the coefficients through an mbarrier per row in flight; in the
//     short-row build the row warp and the consumer warps meet at a named
//     barrier once a row.
//   * Masked rows need no logits, only an all-zero gradient row, written as
//     bulk copies of a zeroed shared-memory block (the copy engine, not the
//     consumers' store path): by a zero warp kept within eight rows of the
//     consumers (long rows), or by the producer as it walks the rows (short
//     rows: one warp fewer leaves 96 registers per thread at two CTAs per
//     SM).
//   * Each row loop reads the mask bytes of 32 of its rows with one ballot
//     and jumps to the next row it handles.
//   * N (valid tokens) is counted by every CTA at start (R bytes from L2);
//     the loss is reduced in fp64: per-warp and per-CTA partials in a fixed
//     row order, then the last CTA (atomic ticket, no spinning) sums them in
//     CTA order.  Same inputs, same device -> bitwise identical results.
//   * Every wait on an mbarrier is bounded (1 s); on timeout the kernel
//     raises RL_DEVERR_TIMEOUT, stops, drains its own bulk copies and
//     exits.  In the short-row build the consumers and the row warp still
//     walk their remaining rows after a timeout, without waiting (every
//     bounded wait then returns at once), so that each meets the others at
//     the named barrier once for every row.  No trap, no unbounded spin.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cmath>
#include <cstring>
#include <map>
#include <mutex>
#include <tuple>

#include "rl_device.cuh"

namespace rl {
namespace {

// The source builds twice.  The default build is the configuration for long
// rows: 16 consumer warps, one CTA per SM, 32 KB chunks.  With RL_SHORT_ROWS
// it builds the one for rows of at most kShortRowBytes: 8 consumer warps,
// two CTAs per SM and 16 KB chunks, so that each SM has two rows in flight
// and one row's per-row latencies (the partials' exchange, the row's scalar
// math) overlap the other's streaming.  The C entry points, compiled in the
// default build only, pick one per call from the row length.
#define RL_INTERNAL __attribute__((visibility("hidden")))  // shared by the two builds only
#ifdef RL_SHORT_ROWS
#define RL_CONSUMER_WARPS 8
#define RL_MIN_CTAS_PER_SM 2
#define RL_CHUNK_BYTES 16384
#define RL_LOSS_KERNEL policy_loss_short_rows_kernel
#define RL_ROWS_NS rl_short_rows
#else
#define RL_LOSS_KERNEL policy_loss_kernel
#define RL_ROWS_NS rl_long_rows
#endif

// Tuning knobs (compile-time; the defaults are the shipped configuration).
#ifndef RL_CHUNK_BYTES
#define RL_CHUNK_BYTES 32768
#endif
#ifndef RL_CONSUMER_WARPS
#define RL_CONSUMER_WARPS 16
#endif
#ifndef RL_RING_SLOTS
#define RL_RING_SLOTS 6
#endif
#ifndef RL_MIN_CTAS_PER_SM
#define RL_MIN_CTAS_PER_SM 1
#endif
// L2 policy of the first load of a streamed row: 1 evict-last, 0 normal.
#ifndef RL_STREAM_KEEP_L2
#define RL_STREAM_KEEP_L2 1
#endif
// Chunks of the next row's first pass that the consumers run before the
// second pass of a row: the time the row warp has for that row's arithmetic.
// RL_LEAD_ALL_VALID applies when no row of the batch is masked (the lead
// widens the reuse distance of the L2 lines kept for pass 2, which masked
// rows' zero writes also compete for); rows of at most RL_FULL_LEAD_CHUNKS
// chunks then lead with the whole next row.
#ifndef RL_LEAD_CHUNKS
#define RL_LEAD_CHUNKS 0
#endif
#ifndef RL_LEAD_ALL_VALID
#ifdef RL_SHORT_ROWS
#define RL_LEAD_ALL_VALID 2
#else
#define RL_LEAD_ALL_VALID 1
#endif
#endif
#ifndef RL_FULL_LEAD_CHUNKS
#ifdef RL_SHORT_ROWS
#define RL_FULL_LEAD_CHUNKS 4
#else
#define RL_FULL_LEAD_CHUNKS 0
#endif
#endif

// How a row's coefficients reach the consumers.  1: the row warp and every
// consumer warp meet at a named barrier once a row (short rows; it wakes the
// consumers sooner and lets them lead with a whole row).  0: an mbarrier per
// row in flight that only the row warp arrives on (long rows, where the
// rendezvous would also hold each of the 16 consumer warps for the slowest).
#ifndef RL_ROW_RENDEZVOUS
#ifdef RL_SHORT_ROWS
#define RL_ROW_RENDEZVOUS 1
#else
#define RL_ROW_RENDEZVOUS 0
#endif
#endif

// A row's last, partly filled chunk.  1: padded in shared memory to a full
// one and taken by the full-chunk routine (short rows, where that routine
// alone in the consumers' loop is 5% faster at V = 32000 fp16).  0: its own
// predicated routine (long rows, where the padding measured 0.2% slower).
#ifndef RL_PAD_TAIL
#ifdef RL_SHORT_ROWS
#define RL_PAD_TAIL 1
#else
#define RL_PAD_TAIL 0
#endif
#endif

// Masked rows' zero gradient: 1 a warp of its own, kept within kZeroLead
// rows of the consumers; 0 the producer writes them as it walks the rows
// (one warp fewer: the short-row build keeps 96 registers per thread).
#ifndef RL_ZERO_WARP
#ifdef RL_SHORT_ROWS
#define RL_ZERO_WARP 0
#else
#define RL_ZERO_WARP 1
#endif
#endif

constexpr int kChunkBytes = RL_CHUNK_BYTES;
constexpr int kSlots = RL_RING_SLOTS;
constexpr int kConsumerWarps = RL_CONSUMER_WARPS;
constexpr int kConsumerThreads = kConsumerWarps * 32;
constexpr int kRowWarp = kConsumerWarps;  // warps: consumers, the row warp, the producer, the zero warp
constexpr int kProducerWarp = kConsumerWarps + 1;
constexpr int kZeroWarp = RL_ZERO_WARP ? kConsumerWarps + 2 : -1;
constexpr int kThreads = kConsumerThreads + (RL_ZERO_WARP ? 96 : 64);
constexpr int kRedWarps = kConsumerWarps + 1;  // consumers and the row warp: token counts and sums
constexpr int kRedThreads = kRedWarps * 32;
constexpr int kLeadChunks = RL_LEAD_CHUNKS;
constexpr int kLeadAllValid = RL_LEAD_ALL_VALID;
constexpr int kFullLeadChunks = RL_FULL_LEAD_CHUNKS;
constexpr bool kRendezvous = RL_ROW_RENDEZVOUS;
constexpr int kVecsPerChunk = kChunkBytes / 16;
constexpr int kVecsPerThread = kVecsPerChunk / kConsumerThreads;
static_assert(kVecsPerChunk % kConsumerThreads == 0, "chunk must split evenly over consumers");
static_assert(kConsumerWarps <= 32, "the row warp takes one consumer partial per lane");
static_assert(kLeadChunks >= 0 && kLeadAllValid >= 0 && kFullLeadChunks >= 0, "chunks of look-ahead");
constexpr int kMaxResidentChunks = (kSlots - 1) / 2;  // two rows + one chunk of look-ahead
constexpr uint32_t kRedBarrier = 1;  // named barrier id (0 is __syncthreads): consumers + row warp
constexpr uint32_t kCoefBarrier = 2;  // named barrier id of the row rendezvous: the same threads
// Zero block the masked rows are copied from (16 KB: with it two CTAs of the
// short-row build fill the SM's 228 KB of shared memory).
constexpr int kZeroBytes = 16384;
constexpr long long kZeroLead = 8;           // rows a zero warp may run ahead of the consumers

// A row's pass-2 coefficients: d_v = 2^x (a0 + a1 x) with x = z log2(e) - cL
// (- cL_lo as well for fp32 logits); the sampled id's element also gets -gy.
struct RowCoef {
  float cL, cL_lo, a0, a1, gy;
};

struct LossSmem {
  alignas(128) unsigned char ring[kSlots][kChunkBytes];
  alignas(128) unsigned char zeros[kZeroBytes];  // source of the masked rows' bulk stores
  unsigned long long full[kSlots];
  unsigned long long empty[kSlots];
  unsigned long long xbar[2];  // a row's consumer partials are in (one arrival per consumer warp)
  unsigned long long cbar[2];  // the row warp is done with a row's partials, coef holds its coefficients
  float4 xpart[2][kConsumerWarps];  // (m, s, t, -) per consumer warp
  float zy[2];                      // the sampled logit, from the thread that holds it (or -inf)
  RowCoef coef[2];
  long long wcount[kThreads / 32];
  long long wseq[kRedWarps];
  double wred[kRedWarps][5];  // per-warp J, pg, kl, H, clipped sums
  int abort;
  int is_last;
  long long pace;  // row the consumers are on (a zero warp keeps within kZeroLead rows of it)
};

struct LossArgs {
  const unsigned char* logits;
  unsigned char* dlogits;
  const long long* ids;
  const float* logp_old;
  const float* ref_logp;
  const unsigned char* mask;
  const float* adv;
  float* logp_out;
  float* entropy_out;
  rl_loss_stats* stats;
  WsHeader* ws;
  WsPartial* partials;
  long long R, T, V;
  long long row_bytes;  // ld * element bytes
  int adv_mode;         // rl_adv_layout
  int group_size, ddof; // RL_ADV_GROUP_REWARDS
  double std_eps;       // RL_ADV_GROUP_REWARDS
  float clip_lo, clip_hi;  // 1 - eps, 1 + eps_high
  float beta, c_ent, grad_scale;
  int agg;              // rl_loss_agg
  double agg_w;         // RL_AGG_TOKEN_SUM_NORM: 1 / agg_norm
  const long long* global_counts;  // device [N, B'] over all ranks, or null (local counts)
  long long v_offset;              // global id of local column 0 (vocabulary shards)
  long long v_total;               // vocabulary size for the id range check
  float4* partials_out;            // shard partials, pass-1 launch
  const float4* shard_partials;    // [n_shards][R] gathered partials, merge launch
  int n_shards;
  float4* row_coef_out;            // merge launch: (cL, a0, a1, gy) per row, or null
};

// ------------------------------------------------------------------ element formats
// Each format reads 16-byte vectors from shared memory.  clamp() floors every
// element at a large negative finite value (keeping NaN), so that a -inf
// logit contributes exp = 0 and 0 * x = 0 instead of 0 * inf = NaN; vmax() is
// the NaN-propagating maximum of a full vector; unpack() widens to fp32.
// The fp32 and bf16 floor is -2^100: its product with log2 e is exact, so in
// a lane whose running maximum is still the floor a floor element gets
// exponent exactly 0 rather than the rounding error of a 1e30-sized product.
constexpr float kFloor = -0x1p100f;

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}

template <int DT>
struct Elem;

template <>
struct Elem<RL_F32> {
  static constexpr int kBytes = 4, kVec = 4;
  static constexpr uint32_t kFloorWord = 0xF1800000u;  // kFloor
  __device__ static float floor_value() { return kFloor; }
  __device__ static void clamp(uint4& w) {
    w.x = __float_as_uint(max_nan(__uint_as_float(w.x), kFloor));
    w.y = __float_as_uint(max_nan(__uint_as_float(w.y), kFloor));
    w.z = __float_as_uint(max_nan(__uint_as_float(w.z), kFloor));
    w.w = __float_as_uint(max_nan(__uint_as_float(w.w), kFloor));
  }
  __device__ static float vmax(const uint4& w) {
    return max_nan(max_nan(__uint_as_float(w.x), __uint_as_float(w.y)),
                   max_nan(__uint_as_float(w.z), __uint_as_float(w.w)));
  }
  __device__ static void unpack(const uint4& w, float (&z)[kVec]) {
    z[0] = __uint_as_float(w.x);
    z[1] = __uint_as_float(w.y);
    z[2] = __uint_as_float(w.z);
    z[3] = __uint_as_float(w.w);
  }
  __device__ static uint4 pack(const float (&z)[kVec]) {
    return make_uint4(__float_as_uint(z[0]), __float_as_uint(z[1]), __float_as_uint(z[2]),
                      __float_as_uint(z[3]));
  }
  __device__ static void store1(unsigned char* p, float v) { *reinterpret_cast<float*>(p) = v; }
};

// Packed two-element NaN-propagating max of bf16 / fp16 pairs.
__device__ __forceinline__ uint32_t max_nan_bf16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ uint32_t max_nan_f16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.NaN.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

template <>
struct Elem<RL_BF16> {
  static constexpr int kBytes = 2, kVec = 8;
  static constexpr uint32_t kFloor2 = 0xF180F180u;  // (-2^100, -2^100) in bf16
  static constexpr uint32_t kFloorWord = kFloor2;
  __device__ static float floor_value() { return kFloor; }
  __device__ static void clamp(uint4& w) {
    w.x = max_nan_bf16x2(w.x, kFloor2);
    w.y = max_nan_bf16x2(w.y, kFloor2);
    w.z = max_nan_bf16x2(w.z, kFloor2);
    w.w = max_nan_bf16x2(w.w, kFloor2);
  }
  __device__ static float vmax(const uint4& w) {
    const uint32_t m = max_nan_bf16x2(max_nan_bf16x2(w.x, w.y), max_nan_bf16x2(w.z, w.w));
    return max_nan(__uint_as_float(m << 16), __uint_as_float(m & 0xffff0000u));
  }
  __device__ static void unpack(const uint4& w, float (&z)[kVec]) {
    const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      z[2 * k] = __uint_as_float(u[k] << 16);
      z[2 * k + 1] = __uint_as_float(u[k] & 0xffff0000u);
    }
  }
  __device__ static uint4 pack(const float (&z)[kVec]) {
    uint32_t u[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      __nv_bfloat162 h = __floats2bfloat162_rn(z[2 * k], z[2 * k + 1]);
      u[k] = *reinterpret_cast<uint32_t*>(&h);
    }
    return make_uint4(u[0], u[1], u[2], u[3]);
  }
  __device__ static void store1(unsigned char* p, float v) {
    *reinterpret_cast<__nv_bfloat16*>(p) = __float2bfloat16_rn(v);
  }
};

template <>
struct Elem<RL_F16> {
  static constexpr int kBytes = 2, kVec = 8;
  static constexpr uint32_t kFloor2 = 0xFBFFFBFFu;  // (-65504, -65504) in fp16
  static constexpr uint32_t kFloorWord = kFloor2;
  __device__ static float floor_value() { return -65504.f; }
  __device__ static void clamp(uint4& w) {
    w.x = max_nan_f16x2(w.x, kFloor2);
    w.y = max_nan_f16x2(w.y, kFloor2);
    w.z = max_nan_f16x2(w.z, kFloor2);
    w.w = max_nan_f16x2(w.w, kFloor2);
  }
  __device__ static float vmax(const uint4& w) {
    const uint32_t m = max_nan_f16x2(max_nan_f16x2(w.x, w.y), max_nan_f16x2(w.z, w.w));
    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&m));
    return max_nan(f.x, f.y);
  }
  __device__ static void unpack(const uint4& w, float (&z)[kVec]) {
    const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&u[k]));
      z[2 * k] = f.x;
      z[2 * k + 1] = f.y;
    }
  }
  __device__ static uint4 pack(const float (&z)[kVec]) {
    uint32_t u[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      __half2 h = __floats2half2_rn(z[2 * k], z[2 * k + 1]);
      u[k] = *reinterpret_cast<uint32_t*>(&h);
    }
    return make_uint4(u[0], u[1], u[2], u[3]);
  }
  __device__ static void store1(unsigned char* p, float v) {
    *reinterpret_cast<__half*>(p) = __float2half_rn(v);
  }
};

// ------------------------------------------------------------------ online statistics
// A partial (m, s, t) over a set of logits z: m = max z, s = sum 2^x,
// t = sum 2^x * x with x = (z - m) * log2(e).  Then for the full row
// lse = m + ln s and H = ln 2 * (log2 s - t / s).  Each thread keeps one
// two-lane (s, t) pair per vector position of a chunk: independent chains.
__device__ __forceinline__ void merge_stats(float& m, float& s, float& t, float m2, float s2,
                                            float t2) {
  if (m2 > m) {
    float tmp = m; m = m2; m2 = tmp;
    tmp = s; s = s2; s2 = tmp;
    tmp = t; t = t2; t2 = tmp;
  }
  if (s2 == 0.f) return;  // empty partner (a NaN s2 falls through and poisons)
  const float d = (m - m2) * kLog2e;
  const float f = ex2_approx(-d);
  s = fmaf(f, s2, s);
  t = fmaf(f, t2 - d * s2, t);
}

struct ThreadStats {
  float m;    // running max, starting at the clamp floor (finite: no -inf cases)
  float nmL;  // -m * log2(e)
  float2 s[kVecsPerThread];
  float2 t[kVecsPerThread];
};

__device__ __forceinline__ void stats_init(ThreadStats& a) {
  a.m = kFloor;
  a.nmL = -kFloor * kLog2e;
#pragma unroll
  for (int q = 0; q < kVecsPerThread; ++q) a.s[q] = a.t[q] = make_float2(0.f, 0.f);
}

// Raise each lane's running max to vm, rescaling its chains.  The decision
// is taken per warp (all lanes rescale when any lane needs to; for the others
// the factor is exactly 1), so the branch never diverges.  Must be called by
// the whole warp.  A NaN vm never raises the max: its NaN enters through x.
__device__ __forceinline__ void raise_max(float vm, ThreadStats& a) {
  if (__any_sync(0xffffffffu, vm > a.m)) {
    const float nm = fmaxf(a.m, vm);
    const float d = (nm - a.m) * kLog2e;  // >= 0 and finite: both are >= the floor
    const float f = ex2_approx(-d);
    const float2 f2 = make_float2(f, f), nd2 = make_float2(-d, -d);
#pragma unroll
    for (int q = 0; q < kVecsPerThread; ++q) {
      a.t[q] = __fmul2_rn(f2, __ffma2_rn(nd2, a.s[q], a.t[q]));
      a.s[q] = __fmul2_rn(f2, a.s[q]);
    }
    a.m = nm;
    a.nmL = -nm * kLog2e;
  }
}

// Pass-1 update with a full chunk: this thread's kVecsPerThread vectors,
// one running-max check for all of them, then independent chains (whole warp).
template <class E>
__device__ __forceinline__ void accumulate_chunk(uint32_t buf, ThreadStats& a) {
  uint4 w[kVecsPerThread];
  float vm = kFloor;
#pragma unroll
  for (int q = 0; q < kVecsPerThread; ++q) {
    w[q] = ld_shared_v4(buf + q * kConsumerThreads * 16);
    E::clamp(w[q]);
    vm = max_nan(vm, E::vmax(w[q]));
  }
  raise_max(vm, a);
  const float2 L2 = make_float2(kLog2e, kLog2e);
  const float2 nmL = make_float2(a.nmL, a.nmL);
#pragma unroll
  for (int q = 0; q < kVecsPerThread; ++q) {
    float z[E::kVec];
    E::unpack(w[q], z);
    float2 s = a.s[q], t = a.t[q];
#pragma unroll
    for (int i = 0; i < E::kVec; i += 2) {
      const float2 x = __ffma2_rn(make_float2(z[i], z[i + 1]), L2, nmL);
      const float2 e = make_float2(ex2_approx(x.x), ex2_approx(x.y));
      s = __fadd2_rn(s, e);
      t = __ffma2_rn(e, x, t);
    }
    a.s[q] = s;
    a.t[q] = t;
  }
}

// Elements nv .. kVec-1 of a vector set to the format's floor: past the end
// of a row they can never raise the running maximum.
template <class E>
__device__ __forceinline__ void fill_floor(uint4& w, int nv) {
  uint32_t u[4] = {w.x, w.y, w.z, w.w};
  constexpr int kPerWord = E::kVec / 4;  // elements per 32-bit word: 1 or 2
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    if (kPerWord * k >= nv)
      u[k] = E::kFloorWord;
    else if (kPerWord == 2 && 2 * k + 1 >= nv)
      u[k] = (u[k] & 0xffffu) | (E::kFloorWord & 0xffff0000u);
  }
  w = make_uint4(u[0], u[1], u[2], u[3]);
}

// Pass-1 update with a row's last, partly filled chunk (whole warp).  Element
// e0 = first + q * kConsumerThreads * kVec starts this thread's vector q; the
// row ends at element nelem.  The same packed chains as a full chunk, with
// the exponentials of elements past the end set to 0 (so they add exactly 0
// to s and t), and vector positions that no lane of the warp holds skipped.
template <class E>
__device__ __forceinline__ void accumulate_chunk_tail(uint32_t buf, int first, int nelem,
                                                      ThreadStats& a) {
  const int rem = nelem - first;  // elements from this thread's vector 0 to the row's end
  uint4 w[kVecsPerThread];
  float vm = kFloor;
#pragma unroll
  for (int q = 0; q < kVecsPerThread; ++q) {
    const int nv = max(0, min(E::kVec, rem - q * kConsumerThreads * E::kVec));
    w[q] = nv > 0 ? ld_shared_v4(buf + q * kConsumerThreads * 16) : make_uint4(0u, 0u, 0u, 0u);
    if (nv < E::kVec) fill_floor<E>(w[q], nv);
    E::clamp(w[q]);
    vm = max_nan(vm, E::vmax(w[q]));
  }
  raise_max(vm, a);
  const float2 L2 = make_float2(kLog2e, kLog2e);
  const float2 nmL = make_float2(a.nmL, a.nmL);
#pragma unroll
  for (int q = 0; q < kVecsPerThread; ++q) {
    const int nv = max(0, min(E::kVec, rem - q * kConsumerThreads * E::kVec));
    if (!__any_sync(0xffffffffu, nv > 0)) continue;  // warp-uniform
    float z[E::kVec];
    E::unpack(w[q], z);
    float2 s = a.s[q], t = a.t[q];
#pragma unroll
    for (int i = 0; i < E::kVec; i += 2) {
      const float2 x = __ffma2_rn(make_float2(z[i], z[i + 1]), L2, nmL);
      const float2 e = make_float2(i < nv ? ex2_approx(x.x) : 0.f, i + 1 < nv ? ex2_approx(x.y) : 0.f);
      s = __fadd2_rn(s, e);
      t = __ffma2_rn(e, x, t);
    }
    a.s[q] = s;
    a.t[q] = t;
  }
}

// A row's last, partly filled chunk made a full one: this thread's vectors
// past the row's end in the ring slot set to the format's floor (elements
// too, where the end cuts a vector), so that the full-chunk routine can take
// it.  They never raise the running maximum, and their exponentials are
// exactly 0 unless the row's maximum lies within ~88 of the floor
// (remove_padding takes their share out then).  Looped, not unrolled: the
// per-row call adds little code to the consumers' loop.
template <class E>
__device__ __forceinline__ void pad_chunk_tail(uint32_t buf, int first, int nelem) {
  const int rem = nelem - first;  // elements from this thread's vector 0 to the row's end
#pragma unroll 1
  for (int q = 0; q < kVecsPerThread; ++q) {
    const int nv = rem - q * kConsumerThreads * E::kVec;
    if (nv < E::kVec) {
      const uint32_t at = buf + q * kConsumerThreads * 16;  // inside the ring slot
      uint4 w = nv > 0 ? ld_shared_v4(at) : make_uint4(0u, 0u, 0u, 0u);
      fill_floor<E>(w, max(nv, 0));
      st_shared_v4(at, w);
    }
  }
  // bulk copies (the async proxy) write the slot again once it is released
  fence_proxy_async_shared();
}

// A row's (M, S, T) with the share of its n_pad padding elements taken out.
// Each entered the first pass as the floor F and added 2^x to S and 2^x x to
// T, with x = F log2 e - M log2 e in the row's frame (the consumers' own
// rounding): 0 unless x is above -126, i.e. unless every logit of the row is
// within ~88 of F (-inf or floor-valued logits).  Only such rows change.
template <class E>
__device__ __forceinline__ void remove_padding(float M, float& S, float& T, int n_pad) {
  const float x = fmaf(E::floor_value(), kLog2e, -M * kLog2e);
  if (n_pad > 0 && x > -127.f) {
    const float e = ex2_approx(x);
    S -= static_cast<float>(n_pad) * e;
    T -= static_cast<float>(n_pad) * e * x;
  }
}

template <class E>
__device__ __forceinline__ float element_of(uint4 w, int i) {
  float z[E::kVec];
  E::unpack(w, z);
  float r = z[0];
#pragma unroll
  for (int k = 1; k < E::kVec; ++k)
    if (k == i) r = z[k];
  return r;
}

// Two-word fp32 arithmetic for the fp32 build's per-row constants:
// s + e == a + b exactly (Knuth's two-sum; __fadd_rn is never contracted).
__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
  s = __fadd_rn(a, b);
  const float bb = __fsub_rn(s, a);
  e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
}
// ln 2 as a head of 15 significant bits, so that e * head is exact for
// |e| < 512, plus the rest (Cody and Waite's split of the constant).
constexpr float kLn2Hi = 45426.0f / 65536.0f;
constexpr float kLn2Lo = static_cast<float>(0.69314718055994530942 - 45426.0 / 65536.0);

// Pass-2 gradient of one vector: d_v = 2^x (a0 + a1 x), x = z log2(e) - cL.
// Without the entropy term (a1 = 0) no clamp is needed: a -inf logit gives
// 2^x = 0 and 0 * a0 = 0.
// fp32 logits (E::kBytes == 4) carry cL in two words, x = (z log2(e) - cL)
// - cL_lo, and take exp2f: their gradient keeps a few fp32 ulps where a
// 16-bit output's rounding would hide the difference.
template <class E, bool kEntropy>
__device__ __forceinline__ void grad_vec(uint4 w, float cL, float cLlo, float a0, float a1,
                                         float (&d)[E::kVec]) {
  if (kEntropy) E::clamp(w);
  float z[E::kVec];
  E::unpack(w, z);
  const float2 L2 = make_float2(kLog2e, kLog2e);
  const float2 ncL = make_float2(-cL, -cL);
  const float2 A0 = make_float2(a0, a0);
#pragma unroll
  for (int i = 0; i < E::kVec; i += 2) {
    float2 x = __ffma2_rn(make_float2(z[i], z[i + 1]), L2, ncL);
    float2 p;
    if constexpr (E::kBytes == 4) {
      x = __fadd2_rn(x, make_float2(-cLlo, -cLlo));
      p = make_float2(exp2f(x.x), exp2f(x.y));
    } else {
      p = make_float2(ex2_approx(x.x), ex2_approx(x.y));
    }
    const float2 r = kEntropy ? __fmul2_rn(p, __ffma2_rn(make_float2(a1, a1), x, A0)) : __fmul2_rn(p, A0);
    d[i] = r.x;
    d[i + 1] = r.y;
  }
}

// Wait for a bulk copy to land regardless of the abort flag (used to drain).
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = global_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_ns() - t0 > kWaitLimitNs) return;
  }
}

__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
__device__ __forceinline__ uint64_t policy_evict_normal() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// Per-row scalars, loaded one row ahead of their use.
struct RowScalars {
  long long y, b;  // sampled id; sequence of the row
  float A, lpo, rf;
  bool valid;
};

// row / T: a 32-bit division when both fit (the 64-bit one is a long
// software sequence, and every consumer thread needs it once per row).
__device__ __forceinline__ long long seq_of(long long row, long long T) {
  if (((row | T) >> 32) == 0)
    return static_cast<long long>(static_cast<uint32_t>(row) / static_cast<uint32_t>(T));
  return row / T;
}

__device__ __forceinline__ RowScalars load_row(const LossArgs& a, long long row) {
  RowScalars r;
  r.valid = false;
  r.y = 0;
  r.b = 0;
  r.A = r.lpo = r.rf = 0.f;
  if (row < a.R) {
    r.valid = a.mask[row] != 0;
    r.y = a.ids[row];
    r.b = seq_of(row, a.T);
    if (a.adv_mode != RL_ADV_GROUP_REWARDS) r.A = a.adv[a.adv_mode == RL_ADV_PER_TOKEN ? row : r.b];
    r.lpo = a.logp_old ? a.logp_old[row] : 0.f;
    r.rf = a.ref_logp ? a.ref_logp[row] : 0.f;
  }
  return r;
}

__device__ __forceinline__ double warp_sum_d(double v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// A CTA's rows are first, first + stride, first + 2 stride, ... (below R).
// A warp walks the ones whose mask byte is nonzero (kValid) or zero
// (!kValid) a window of 32 at a time: lane k reads the byte of row
// base + k * stride and one ballot gives the window's rows, so a run of
// skipped rows costs one load latency per 32 rows instead of one per row.
// next() returns the next such row, or R after the last; whole warp.
template <bool kValid>
struct RowWalk {
  long long base;
  uint32_t bits;
  __device__ RowWalk(long long first, long long stride) : base(first - 32 * stride), bits(0u) {}
  __device__ __forceinline__ long long next(const unsigned char* mask, long long stride, long long R,
                                            int lane) {
    while (bits == 0u) {
      if (base >= R) return R;
      base += 32 * stride;
      const long long r = base + lane * stride;
      bits = __ballot_sync(0xffffffffu, r < R && ((mask[r] != 0) == kValid));
    }
    const int k = __ffs(bits) - 1;
    bits &= bits - 1u;
    return base + k * stride;
  }
};

// Every row first, first + stride, ... (below R) in order, with its mask
// bit: one ballot per window of 32 rows.  next() returns the next row (R
// after the last) and whether it is valid; whole warp.
struct RowScan {
  long long base;
  uint32_t bits;
  int i;
  __device__ RowScan(long long first, long long stride) : base(first - 32 * stride), bits(0u), i(32) {}
  __device__ __forceinline__ long long next(const unsigned char* mask, long long stride, long long R,
                                            int lane, bool& valid) {
    if (i == 32) {
      base += 32 * stride;
      if (base >= R) {
        valid = false;
        return R;
      }
      const long long r = base + lane * stride;
      bits = __ballot_sync(0xffffffffu, r < R && mask[r] != 0);
      i = 0;
    }
    const long long row = base + i * stride;
    valid = (bits >> i) & 1u;
    ++i;
    return row < R ? row : R;
  }
};

// Nonzero bytes of mask[begin, begin + n), counted by one warp (every lane
// gets the count).
__device__ __forceinline__ int warp_count_mask(const unsigned char* m, long long n, int lane) {
  int c = 0;
  long long i0 = 0;
  if (((reinterpret_cast<uintptr_t>(m)) & 15) == 0) {
    const long long nv = n >> 4;
    const uint4* mv = reinterpret_cast<const uint4*>(m);
    for (long long i = lane; i < nv; i += 32) {
      const uint4 w = __ldg(mv + i);
      c += (__popc(__vcmpne4(w.x, 0u)) + __popc(__vcmpne4(w.y, 0u)) +
            __popc(__vcmpne4(w.z, 0u)) + __popc(__vcmpne4(w.w, 0u))) >> 3;
    }
    i0 = nv << 4;
  }
  for (long long i = i0 + lane; i < n; i += 32) c += m[i] != 0;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
  return c;
}

// Group-relative advantage of sequence b from the rewards (one warp, fp64,
// the same arithmetic as rl_group_advantages): (R_b - mean) / (std + eps).
__device__ __forceinline__ float warp_group_advantage(const LossArgs& a, long long b, int lane) {
  const int G = a.group_size;
  const float* r = a.adv + (b / G) * G;
  double sum = 0.0;
  for (int j = lane; j < G; j += 32) sum += static_cast<double>(r[j]);
  const double mean = warp_sum_d(sum) / G;
  double sq = 0.0;
  for (int j = lane; j < G; j += 32) {
    const double d = static_cast<double>(r[j]) - mean;
    sq += d * d;
  }
  const double std = sqrt(warp_sum_d(sq) / (G - a.ddof));
  const double inv = 1.0 / (std + a.std_eps);
  return static_cast<float>((static_cast<double>(a.adv[b]) - mean) * inv);
}

// ------------------------------------------------------------------ the kernel
// Where a row's sampled id sits, for the consumer thread that holds it:
// chunk cy and, in jv, vector jv / kVec of the chunk and element jv % kVec
// of the vector.  cy = -1 on every other thread, and everywhere when the id
// is not one of this launch's columns.
struct IdPos {
  int cy, jv;
};

template <int kElemsPerChunk, int kVec>
__device__ __forceinline__ IdPos id_pos(const LossArgs& a, long long y, int tid) {
  IdPos p;
  p.cy = -1;
  p.jv = 0;
  const long long yl = y - a.v_offset;  // column of y in this shard
  if (yl >= 0 && yl < a.V) {
    const int off = static_cast<int>(yl);
    const int jv = off % kElemsPerChunk;  // element within the chunk
    if ((jv / kVec) % kConsumerThreads == tid) {
      p.cy = off / kElemsPerChunk;
      p.jv = jv;
    }
  }
  return p;
}

// Per-sequence quantities of a warp's current sequence.
struct SeqCache {
  long long b;
  int L;    // valid tokens of the sequence (seq-mean-token-mean)
  float A;  // group advantage from the rewards
};

// Merge of per-shard statistics (vocabulary shards, merge launch): shard
// order over the lanes, then a fixed shuffle tree; every lane returns lane
// 0's bits.  Whole warp.
__device__ __forceinline__ void merge_shards(const LossArgs& a, long long row, int lane, float& M,
                                             float& S, float& Tt, float& zyr) {
  M = -INFINITY;
  S = Tt = 0.f;
  zyr = -INFINITY;
  for (int k = lane; k < a.n_shards; k += 32) {
    const float4 P = __ldg(&a.shard_partials[static_cast<long long>(k) * a.R + row]);
    merge_stats(M, S, Tt, P.x, P.y, P.z);
    zyr = max_nan(zyr, P.w);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, M, o);
    const float s2 = __shfl_xor_sync(0xffffffffu, S, o);
    const float t2 = __shfl_xor_sync(0xffffffffu, Tt, o);
    merge_stats(M, S, Tt, m2, s2, t2);
    zyr = max_nan(zyr, __shfl_xor_sync(0xffffffffu, zyr, o));
  }
  M = __shfl_sync(0xffffffffu, M, 0);
  S = __shfl_sync(0xffffffffu, S, 0);
  Tt = __shfl_sync(0xffffffffu, Tt, 0);
  zyr = __shfl_sync(0xffffffffu, zyr, 0);
}

// Sum of (m, s, t) partials over the warp: the maximum first, then each
// lane's sums rescaled to it and added.  Lane 0 holds the result (every lane
// gets it with `bcast`).  A partial with s = 0 adds exactly 0; a NaN s or t
// poisons the sum.
__device__ __forceinline__ void warp_stats(float& m, float& s, float& t, bool bcast) {
  float M;
  asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(M) : "f"(m));
  const float d = (M - m) * kLog2e;  // >= 0, finite: every m is at least the floor
  const float f = ex2_approx(-d);
  t = f * fmaf(-d, s, t);
  s = f * s;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    s += __shfl_xor_sync(0xffffffffu, s, o);
    t += __shfl_xor_sync(0xffffffffu, t, o);
  }
  m = M;
  if (bcast) {
    s = __shfl_sync(0xffffffffu, s, 0);
    t = __shfl_sync(0xffffffffu, t, 0);
  }
}

// A row's loss terms and the coefficients of its gradient.
struct RowVals {
  RowCoef cf;
  float J, pg, kl, H, logp;
  double w_row;
  bool clipped, y_ok;
};

// From a row's softmax statistics (M, S, Tt, z_y) to its loss terms and the
// coefficients of its gradient.  Whole warp: every lane computes the same
// values from the same inputs.  16-bit logits take the fast hardware log2,
// exp and division for lse, the ratio and the entropy (errors near 1e-6
// relative, far below what a 16-bit gradient or the loss's tolerance can
// show); fp32 logits keep the accurate two-word path.
template <int DT>
__device__ __forceinline__ RowVals row_values(const LossArgs& a, const RowScalars& rs, SeqCache& cache,
                                              long long Bp, float sc, float M, float S, float Tt,
                                              float zyr, int lane) {
  RowVals v;
  // per-sequence quantities, recomputed when the sequence changes
  const long long bseq = rs.b;
  if (bseq != cache.b) {
    cache.b = bseq;
    if (a.agg == RL_AGG_SEQ_MEAN_TOKEN_MEAN) cache.L = warp_count_mask(a.mask + bseq * a.T, a.T, lane);
    if (a.adv_mode == RL_ADV_GROUP_REWARDS) cache.A = warp_group_advantage(a, bseq, lane);
  }
  // loss weight of this token and the gradient scale of its row
  v.w_row = 1.0;  // token mean: the 1/N is applied once, at the end
  float sc_row = sc;
  if (a.agg != RL_AGG_TOKEN_MEAN) {
    v.w_row = a.agg == RL_AGG_SEQ_MEAN_TOKEN_MEAN ? 1.0 / (static_cast<double>(Bp) * cache.L)
            : a.agg == RL_AGG_SEQ_MEAN_TOKEN_SUM  ? 1.0 / static_cast<double>(Bp)
                                                   : a.agg_w;
    sc_row = static_cast<float>(static_cast<double>(a.grad_scale) * v.w_row);
  }
  const long long y = rs.y;
  v.y_ok = (y >= 0) && (y < a.v_total);
  const float zv = v.y_ok ? zyr : __int_as_float(0x7fc00000);
  // lse = M + ln S, logp = z_y - lse and cL = M log2(e) + log2 S (pass 2's
  // exponent offset).  fp32 logits keep logp and cL in two words: with
  // S = m 2^e (m in [0.5, 1)), log2 S = e + log2 m and ln S = e ln 2 + ln m,
  // summed without rounding away the bits a single fp32 lse (|lse| ~ 10)
  // would lose; 16-bit logits need no more than one word.
  float log2S, logp, lp_lo = 0.f, cL, cL_lo = 0.f, TtS;
  if constexpr (DT == RL_F32) {
    int e2;
    const float m2 = frexpf(S, &e2);
    const float l2m = log2f(m2), ef = static_cast<float>(e2);
    log2S = ef + l2m;
    float s1, r1, s2, r2, s3, r3;
    two_sum(zv, -M, s1, r1);
    two_sum(s1, -ef * kLn2Hi, s2, r2);
    two_sum(s2, -kLn2 * l2m, s3, r3);
    logp = s3;
    lp_lo = (r1 + r2) + (r3 - ef * kLn2Lo);
    const float p1 = M * kLog2e, q1 = fmaf(M, kLog2e, -p1);  // M log2(e) = p1 + q1 exactly
    float c1, f1, c2, f2;
    two_sum(p1, ef, c1, f1);
    two_sum(c1, l2m, c2, f2);
    cL = c2;
    cL_lo = (f1 + f2) + q1;
    TtS = Tt / S;
  } else {
    log2S = __log2f(S);  // S >= 1: the row's maximum contributes 2^0
    TtS = __fdividef(Tt, S);
    logp = zv - fmaf(log2S, kLn2, M);
    cL = fmaf(M, kLog2e, log2S);
  }
  v.H = kLn2 * (log2S - TtS);
  v.logp = logp;

  // per-token objective and its derivative with respect to logp
  const float A = a.adv_mode == RL_ADV_GROUP_REWARDS ? cache.A : rs.A;
  float r = 1.f;
  if (a.logp_old) {
    if constexpr (DT == RL_F32) {  // exp of the two-word difference
      float u, ue;
      two_sum(logp, -rs.lpo, u, ue);
      const float r0 = expf(u);
      r = fmaf(r0, ue + lp_lo, r0);
    } else {
      r = __expf(logp - rs.lpo);
    }
  }
  const float rA = r * A;
  v.pg = fminf(rA, fminf(fmaxf(r, a.clip_lo), a.clip_hi) * A);
  v.clipped = (A > 0.f && r > a.clip_hi) || (A < 0.f && r < a.clip_lo);
  const float dpg = v.clipped ? 0.f : rA;
  float dkl = 0.f;
  v.kl = 0.f;
  if (a.ref_logp) {
    if constexpr (DT == RL_F32) {
      float d, de;
      two_sum(rs.rf, -logp, d, de);
      de -= lp_lo;
      const float em = expm1f(d);
      dkl = fmaf(em + 1.f, de, em);
      v.kl = (em - d) + fmaf(em, de, 0.f);
    } else {
      const float d = rs.rf - logp;
      dkl = expm1f(d);
      v.kl = dkl - d;
    }
  }
  v.J = v.pg - a.beta * v.kl + a.c_ent * v.H;
  float g = dpg + a.beta * dkl;
  if (logp != logp) {  // NaN logp (bad id or NaN logits): poison the row
    v.J = logp;
    g = logp;
  }
  // pass 2: dz_v = sc [g (p_v - [v == y]) + c_ent p_v (ln p_v + H)]
  // with x_v = z_v log2(e) - cL:  p_v = 2^x_v, ln p_v = x_v ln 2
  v.cf.cL = cL;
  v.cf.cL_lo = cL_lo;
  v.cf.a0 = sc_row * fmaf(a.c_ent, v.H, g);
  v.cf.a1 = sc_row * a.c_ent * kLn2;
  v.cf.gy = sc_row * g;
  return v;
}

// Lane 0 adds the row's terms to `acc` and writes its per-row outputs
// (logp, entropy, row coefficients).
__device__ __forceinline__ void row_book(const LossArgs& a, long long row, const RowVals& v, int lane,
                                         double* acc, unsigned int& err) {
  if (lane != 0) return;
  acc[0] += a.agg == RL_AGG_TOKEN_MEAN ? static_cast<double>(v.J) : v.w_row * v.J;
  acc[1] += v.pg;
  acc[2] += v.kl;
  acc[3] += v.H;
  acc[4] += v.clipped ? 1.0 : 0.0;
  if (!v.y_ok) err |= RL_DEVERR_ID_RANGE;
  if (a.logp_out) a.logp_out[row] = v.logp;
  if (a.entropy_out) a.entropy_out[row] = v.H;
  if (a.row_coef_out) a.row_coef_out[row] = make_float4(v.cf.cL, v.cf.a0, v.cf.a1, v.cf.gy);
}

// A masked row needs no logits, only an all-zero gradient row: bulk copies
// of a zeroed shared-memory block (the copy engine, not the consumers' store
// path) plus plain stores for a row end that is not a multiple of 16 bytes,
// and zero per-row outputs.  Whole warp.
template <class E, int kMode>
__device__ __forceinline__ void zero_row(const LossArgs& a, uint32_t zeros, long long row, int nelem,
                                         uint64_t pol, int lane) {
  if (a.dlogits) {
    const long long nb16 = static_cast<long long>(nelem) * E::kBytes & ~15LL;  // bulk part of the row
    unsigned char* d = a.dlogits + row * a.row_bytes;
    if (lane == 0) {
      for (long long off = 0; off < nb16; off += kZeroBytes)
        bulk_store(d + off, zeros, static_cast<uint32_t>(min(static_cast<long long>(kZeroBytes), nb16 - off)),
                   pol);
      bulk_commit();
    }
    for (long long e = nb16 / E::kBytes + lane; e < nelem; e += 32) E::store1(d + e * E::kBytes, 0.f);
  }
  if (lane == 0) {
    if (a.logp_out) a.logp_out[row] = 0.f;
    if (a.entropy_out) a.entropy_out[row] = 0.f;
    if (kMode >= 2 && a.row_coef_out) a.row_coef_out[row] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
}

// kStream: rows are streamed twice through the ring (second pass from L2);
// otherwise each row stays in the ring for both passes.
// kMode: 0 the whole loss; 1 (vocabulary shard) pass 1 only, writing each
// row's partial statistics; 2 (vocabulary shard) merge the gathered shard
// partials instead of pass 1, then the loss and this shard's gradient; 3 the
// merge of mode 2 with no columns at all (each row's gradient coefficients
// are its only per-row output besides logp and entropy): nothing is shared
// between the warps of a row then, so every consumer warp takes its own rows.
//
// Roles (modes 0-2).  The consumer warps stream the ring: pass 1 of a row,
// then each warp publishes one (m, s, t) partial.  The row warp merges the
// partials and turns them into the row's loss terms and pass-2
// coefficients; meanwhile the consumers already run the first kLead chunks
// of the next row's pass 1, then pass 2 of the row, then the rest of the
// next row's pass 1.  So a row's merge and scalar arithmetic (a long
// dependent chain) overlap streaming instead of stalling every consumer
// warp, and run once per row instead of once per warp.  The producer issues
// the chunks in exactly that order; xbar[b] (consumers -> row warp) and
// cbar[b] (row warp -> consumers) alternate between two rows in flight.
template <int DT, bool kStream, int kMode, bool kEnt>
__global__ void __launch_bounds__(kThreads, RL_MIN_CTAS_PER_SM) RL_LOSS_KERNEL(const LossArgs a) {
  using E = Elem<DT>;
  constexpr int kVec = E::kVec;
  constexpr int kChunkElems = kChunkBytes / E::kBytes;

  extern __shared__ __align__(128) unsigned char smem_raw[];
  LossSmem& sm = *reinterpret_cast<LossSmem*>(smem_raw);
  volatile int* abort_flag = &sm.abort;

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const long long cid = blockIdx.x, ncl = gridDim.x;

  if (tid == 0) {
    for (int s = 0; s < kSlots; ++s) {
      mbar_init(smem_addr(&sm.full[s]), 1);
      mbar_init(smem_addr(&sm.empty[s]), kConsumerWarps);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_addr(&sm.xbar[b]), kConsumerWarps);
      mbar_init(smem_addr(&sm.cbar[b]), 1);
      sm.zy[b] = -INFINITY;
    }
    sm.abort = 0;
    sm.is_last = 0;
    sm.pace = -1;
    fence_mbar_init();
  }
  __syncthreads();
  // Launched with programmatic stream serialisation: the set-up above overlaps
  // the previous kernel (e.g. the advantages); nothing in global memory is
  // read before that kernel has finished.
  grid_dependency_wait();

  const int nelem = static_cast<int>(a.V);
  const long long row_bytes16 = (static_cast<long long>(nelem) * E::kBytes + 15) & ~15LL;
  const int nchunks = static_cast<int>((row_bytes16 + kChunkBytes - 1) / kChunkBytes);
  constexpr bool kTwoPass = kStream && kMode == 0;  // pass-2 chunks come through the ring again

  // N = number of valid tokens; every CTA counts the whole mask.
  long long cnt = 0;
  {
    long long i0 = 0;
    if ((reinterpret_cast<uintptr_t>(a.mask) & 15) == 0) {
      const long long nv = a.R >> 4;
      const uint4* mv = reinterpret_cast<const uint4*>(a.mask);
      for (long long i = tid; i < nv; i += kThreads) {
        const uint4 w = __ldg(mv + i);
        cnt += (__popc(__vcmpne4(w.x, 0u)) + __popc(__vcmpne4(w.y, 0u)) +
                __popc(__vcmpne4(w.z, 0u)) + __popc(__vcmpne4(w.w, 0u))) >> 3;
      }
      i0 = nv << 4;
    }
    for (long long i = i0 + tid; i < a.R; i += kThreads) cnt += a.mask[i] != 0;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
    if (lane == 0) sm.wcount[warp] = cnt;
    __syncthreads();
    cnt = 0;
    for (int w = 0; w < kThreads / 32; ++w) cnt += sm.wcount[w];
  }
  const long long N_local = cnt;
  // When no row is masked, a streamed row's second pass runs in reverse chunk
  // order (its last chunks, loaded most recently, are read again first) and
  // the consumers lead with kLeadAllValid chunks, or the whole row for rows
  // of at most kFullLeadChunks chunks; with masked rows, whose zero writes
  // also pass through L2, in load order with kLeadChunks.
  const bool all_valid = N_local == a.R;
  const bool rev = kTwoPass && all_valid;
  const int lead_chunks = !all_valid                                   ? kLeadChunks
                          : kFullLeadChunks > 0 && nchunks <= kFullLeadChunks ? nchunks
                                                                       : kLeadAllValid;
  // Rows whose coefficients reach the consumers through the rendezvous.  Its
  // participants never leave their row loops early: after a timeout every
  // bounded wait returns at once, so each of them still meets the others
  // once for every row of the CTA and the barrier cannot be left waiting.
  constexpr bool kMeet = kRendezvous && (kMode == 0 || kMode == 2);

  if (warp == kProducerWarp) {
    // ---------------------------------------------------------------- producer
    // The warp walks this CTA's rows; lane 0 issues the valid rows' copies in
    // the order the consumers take them.  Without a zero warp it also writes
    // the masked rows as it passes them: the ring keeps it within a few
    // chunks of the consumers, so those writes spread over the launch.
    if (!RL_ZERO_WARP) {
      for (int i = lane; i < kZeroBytes / 16; i += 32)
        reinterpret_cast<uint4*>(sm.zeros)[i] = make_uint4(0u, 0u, 0u, 0u);
      fence_proxy_async_shared();
      __syncwarp();
    }
    const uint64_t pol_last = RL_STREAM_KEEP_L2 ? policy_evict_last() : policy_evict_normal();
    const uint64_t pol_first = policy_evict_first();
    uint32_t it = 0;
    bool stop = false;
    auto issue = [&](long long row, int c0, int c1, uint64_t pol, bool reverse) {
      if (lane != 0 || stop) return;
      const unsigned char* src = a.logits + row * a.row_bytes;
      for (int i = c0; i < c1; ++i, ++it) {
        const int c = reverse ? c1 - 1 - (i - c0) : i;
        const uint32_t slot = it % kSlots, round = it / kSlots;
        if (round > 0 && !wait_bounded<false>(smem_addr(&sm.empty[slot]), (round - 1) & 1, abort_flag)) {
          stop = true;
          return;
        }
        if (*abort_flag) {
          stop = true;
          return;
        }
        const uint32_t bytes = static_cast<uint32_t>(
            min(static_cast<long long>(kChunkBytes), row_bytes16 - static_cast<long long>(c) * kChunkBytes));
        const uint32_t fb = smem_addr(&sm.full[slot]);
        mbar_arrive_expect_tx(fb, bytes);
        bulk_load(smem_addr(sm.ring[slot]), src + static_cast<long long>(c) * kChunkBytes, bytes, fb, pol);
      }
    };
    long long prev = -1;  // two-pass order: the valid row whose second pass is still to issue
    auto valid_row = [&](long long row) {
      if constexpr (kTwoPass) {
        if (prev >= 0) {
          const int lead = min(nchunks, lead_chunks);
          issue(row, 0, lead, pol_last, false);
          issue(prev, 0, nchunks, pol_first, rev);
          issue(row, lead, nchunks, pol_last, false);
        } else {
          issue(row, 0, nchunks, pol_last, false);
        }
        prev = row;
      } else if (kMode != 3) {
        issue(row, 0, nchunks, pol_first, false);
      }
      stop = __shfl_sync(0xffffffffu, stop, 0);
    };
    if constexpr (RL_ZERO_WARP) {
      RowWalk<true> walk(cid, ncl);
      if (kMode != 3)
        for (long long row = walk.next(a.mask, ncl, a.R, lane); row < a.R && !stop;
             row = walk.next(a.mask, ncl, a.R, lane))
          valid_row(row);
    } else {
      const uint64_t pol_zero = policy_evict_first();
      RowScan scan(cid, ncl);
      while (!stop) {
        bool valid;
        const long long row = scan.next(a.mask, ncl, a.R, lane, valid);
        if (row >= a.R) break;
        if (valid)
          valid_row(row);
        else
          zero_row<E, kMode>(a, smem_addr(sm.zeros), row, nelem, pol_zero, lane);
      }
    }
    if (kTwoPass && prev >= 0) issue(prev, 0, nchunks, pol_first, rev);
    if (lane == 0 && stop && nchunks > 0) {  // let every copy already issued land before this CTA can exit
      for (uint32_t k = it > kSlots ? it - kSlots : 0; k < it; ++k)
        drain_wait(smem_addr(&sm.full[k % kSlots]), (k / kSlots) & 1);
    }
    if (!RL_ZERO_WARP && lane == 0) bulk_wait_all();  // the zero block is read until the last copy is done
    return;
  }

  if (warp == kZeroWarp) {
    // ---------------------------------------------------------------- zero warp
    // Writes the masked rows while the consumers work on the valid rows, so
    // their stores overlap the valid rows' arithmetic.  It keeps within
    // kZeroLead rows of the consumers, so the writes stay spread over the
    // launch instead of arriving as one burst at its start.
    for (int i = lane; i < kZeroBytes / 16; i += 32)
      reinterpret_cast<uint4*>(sm.zeros)[i] = make_uint4(0u, 0u, 0u, 0u);
    fence_proxy_async_shared();
    __syncwarp();
    const uint64_t pol = policy_evict_first();
    const volatile long long* pace = &sm.pace;
    RowWalk<false> walk(cid, ncl);
    for (long long row = walk.next(a.mask, ncl, a.R, lane); row < a.R; row = walk.next(a.mask, ncl, a.R, lane)) {
      if (kMode != 3 && *pace < row - kZeroLead * ncl) {  // bounded wait, then go on
        const uint64_t t0 = global_ns();
        while (*pace < row - kZeroLead * ncl && global_ns() - t0 < kWaitLimitNs) __nanosleep(500);
      }
      zero_row<E, kMode>(a, smem_addr(sm.zeros), row, nelem, pol, lane);
    }
    if (lane == 0) bulk_wait_all();  // the block is read until the last copy is done
    return;
  }

  // ------------------------------------------------------------------ consumers and the row warp
  // Data parallel over ranks: the means run over every rank's tokens.
  const long long N = a.global_counts ? a.global_counts[0] : N_local;
  const float sc = N > 0 ? static_cast<float>(static_cast<double>(a.grad_scale) / static_cast<double>(N)) : 0.f;
  const bool seq_agg = a.agg == RL_AGG_SEQ_MEAN_TOKEN_MEAN || a.agg == RL_AGG_SEQ_MEAN_TOKEN_SUM;
  long long Bp = 0;  // sequences with at least one valid token
  if (seq_agg && a.global_counts) {
    Bp = a.global_counts[1];
  } else if (seq_agg) {
    const long long nseq = a.R / a.T;
    long long nb = 0;
    for (long long b = warp; b < nseq; b += kRedWarps) nb += warp_count_mask(a.mask + b * a.T, a.T, lane) > 0;
    if (lane == 0) sm.wseq[warp] = nb;
    named_barrier(kRedBarrier, kRedThreads);
    for (int w = 0; w < kRedWarps; ++w) Bp += sm.wseq[w];
  }

  unsigned int err = 0;
  double wacc[5] = {0.0, 0.0, 0.0, 0.0, 0.0};  // this warp's sums (lane 0)

  if constexpr (kMode == 3) {
    // ---------------------------------------------------------------- coefficient-only merge
    // Each consumer warp takes its own rows; the row warp has none.
    if (warp < kConsumerWarps) {
      const long long rstride = ncl * kConsumerWarps;
      RowWalk<true> walk(cid * kConsumerWarps + warp, rstride);
      SeqCache cache{-1, 0, 0.f};
      long long nrow = walk.next(a.mask, rstride, a.R, lane);
      RowScalars cur = load_row(a, nrow);
      for (long long row = nrow; row < a.R; row = nrow) {
        nrow = walk.next(a.mask, rstride, a.R, lane);
        const RowScalars rs = cur;
        cur = load_row(a, nrow);
        float M, S, Tt, zyr;
        merge_shards(a, row, lane, M, S, Tt, zyr);
        row_book(a, row, row_values<DT>(a, rs, cache, Bp, sc, M, S, Tt, zyr, lane), lane, wacc, err);
      }
    }
  } else if (warp == kRowWarp) {
    // ---------------------------------------------------------------- row warp
    RowWalk<true> walk(cid, ncl);
    SeqCache cache{-1, 0, 0.f};
    long long row = walk.next(a.mask, ncl, a.R, lane);
    RowScalars rs = load_row(a, row);
    for (uint32_t k = 0; row < a.R; ++k) {
      const long long nrow = walk.next(a.mask, ncl, a.R, lane);
      const RowScalars nrs = load_row(a, nrow);  // next row's scalars, in flight during this row
      const uint32_t b = k & 1;
      float M, S, Tt, zyr;
      if constexpr (kMode < 2) {
        // the consumer warps' partials of this row
        if (!wait_bounded<false>(smem_addr(&sm.xbar[b]), (k >> 1) & 1, abort_flag) && !kMeet) break;
        const float4 P = lane < kConsumerWarps ? sm.xpart[b][lane] : make_float4(kFloor, 0.f, 0.f, 0.f);
        M = P.x;
        S = P.y;
        Tt = P.z;
        warp_stats(M, S, Tt, true);
        if (RL_PAD_TAIL) remove_padding<E>(M, S, Tt, nchunks * kChunkElems - nelem);
        zyr = sm.zy[b];
        __syncwarp();
        if (lane == 0) sm.zy[b] = -INFINITY;  // for the row after next (written after cbar[b] below)
      } else {
        // consumers took row k - 2's coefficients before coef[b] is rewritten
        // (the rendezvous of row k - 1 already orders that)
        if (!kMeet && k >= 2 && !wait_bounded<false>(smem_addr(&sm.xbar[b]), ((k - 2) >> 1) & 1, abort_flag))
          break;
        merge_shards(a, row, lane, M, S, Tt, zyr);
      }
      if constexpr (kMode == 1) {  // this shard's statistics of the row, for the exchange
        if (lane == 0) {
          a.partials_out[row] = make_float4(M, S, Tt, zyr);
          mbar_arrive(smem_addr(&sm.cbar[b]));
        }
      } else {
        const RowVals v = row_values<DT>(a, rs, cache, Bp, sc, M, S, Tt, zyr, lane);
        // the consumers' coefficients first, the bookkeeping after
        if constexpr (kMeet) {
          if (lane == 0) sm.coef[b] = v.cf;
          __syncwarp();
          named_barrier(kCoefBarrier, kRedThreads);
        } else if (lane == 0) {
          sm.coef[b] = v.cf;
          mbar_arrive(smem_addr(&sm.cbar[b]));
        }
        row_book(a, row, v, lane, wacc, err);
      }
      row = nrow;
      rs = nrs;
    }
  } else {
    // ---------------------------------------------------------------- consumers
    uint32_t it = 0;  // position in the ring
    // pass 1 over chunks [c0, c1) of a row: this thread's online statistics
    auto pass1 = [&](int c0, int c1, ThreadStats& st, float& zy, const IdPos& p) {
      for (int c = c0; c < c1; ++c) {
        const uint32_t k = it++, slot = k % kSlots;
        wait_bounded<false>(smem_addr(&sm.full[slot]), (k / kSlots) & 1, abort_flag);
        const uint32_t buf = smem_addr(sm.ring[slot]) + tid * 16;
        const int e0 = c * kChunkElems;
        if (RL_PAD_TAIL) {
          if (e0 + kChunkElems > nelem) pad_chunk_tail<E>(buf, e0 + tid * kVec, nelem);
          accumulate_chunk<E>(buf, st);
        } else if (e0 + kChunkElems <= nelem) {
          accumulate_chunk<E>(buf, st);
        } else {
          accumulate_chunk_tail<E>(buf, e0 + tid * kVec, nelem, st);
        }
        if (c == p.cy) zy = element_of<E>(ld_shared_v4(smem_addr(sm.ring[slot]) + p.jv / kVec * 16), p.jv % kVec);
        if (kStream || kMode == 1) {  // read again from L2 in pass 2 (or no pass 2): free it now
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_addr(&sm.empty[slot]));
        }
      }
    };
    // this thread's statistics folded into one (m, s, t)
    auto fold = [&](const ThreadStats& st, float& m, float& s, float& t) {
      m = st.m;
      s = t = 0.f;
#pragma unroll
      for (int q = 0; q < kVecsPerThread; ++q) {
        s += st.s[q].x + st.s[q].y;
        t += st.t[q].x + st.t[q].y;
      }
    };
    // the warp's partial of row k for the row warp (after row k - 2's partials
    // were taken); (m0, s0, t0): this thread's fold of the row's first chunks
    auto publish = [&](uint32_t k, const ThreadStats& st, float m0, float s0, float t0, float zy,
                       const IdPos& p) {
      float m, s, t;
      fold(st, m, s, t);
      merge_stats(m, s, t, m0, s0, t0);
      warp_stats(m, s, t, false);
      const uint32_t b = k & 1;
      // (with the rendezvous, this warp's meeting for row k - 1 already orders that)
      if (!kMeet && k >= 2) wait_bounded<false>(smem_addr(&sm.cbar[b]), ((k - 2) >> 1) & 1, abort_flag);
      if (p.cy >= 0) sm.zy[b] = zy;
      __syncwarp();
      if (lane == 0) {
        sm.xpart[b][warp] = make_float4(m, s, t, 0.f);
        mbar_arrive(smem_addr(&sm.xbar[b]));
      }
    };
    // pass 2 of row `row` (the k-th of this CTA; resident rows start at ring position `base`)
    auto pass2 = [&](long long row, uint32_t k, uint32_t base, const IdPos& p) {
      const uint32_t b = k & 1;
      if constexpr (kMeet)
        named_barrier(kCoefBarrier, kRedThreads);
      else
        wait_bounded<false>(smem_addr(&sm.cbar[b]), (k >> 1) & 1, abort_flag);
      const RowCoef cf = sm.coef[b];
      if (!kMeet && kMode == 2) {  // coef[b] taken: the row warp may rewrite it for row k + 2
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_addr(&sm.xbar[b]));
      }
      unsigned char* drow = a.dlogits ? a.dlogits + row * a.row_bytes : nullptr;
      for (int i = 0; i < nchunks; ++i) {
        const int c = rev ? nchunks - 1 - i : i;
        uint32_t slot;
        if (kStream || kMode == 2) {
          const uint32_t kk = it++;
          slot = kk % kSlots;
          wait_bounded<false>(smem_addr(&sm.full[slot]), (kk / kSlots) & 1, abort_flag);
        } else {
          slot = (base + c) % kSlots;
        }
        if (drow) {
          const uint32_t buf = smem_addr(sm.ring[slot]);
          const int c0 = c * kChunkElems;
          unsigned char* dst = drow + static_cast<long long>(c0 + tid * kVec) * E::kBytes;
          if (c0 + kChunkElems <= nelem) {
#pragma unroll
            for (int q = 0; q < kVecsPerThread; ++q) {
              float d[kVec];
              const uint4 w = ld_shared_v4(buf + (tid + q * kConsumerThreads) * 16);
              grad_vec<E, kEnt>(w, cf.cL, cf.cL_lo, cf.a0, cf.a1, d);
              st_global_cs_v4(dst + q * kConsumerThreads * 16, E::pack(d));
            }
          } else {
#pragma unroll
            for (int q = 0; q < kVecsPerThread; ++q) {
              const int e0 = c0 + (tid + q * kConsumerThreads) * kVec;
              if (e0 < nelem) {
                float d[kVec];
                const uint4 w = ld_shared_v4(buf + (tid + q * kConsumerThreads) * 16);
                grad_vec<E, kEnt>(w, cf.cL, cf.cL_lo, cf.a0, cf.a1, d);
                unsigned char* o = dst + q * kConsumerThreads * 16;
                if (nelem - e0 >= kVec) {
                  st_global_cs_v4(o, E::pack(d));
                } else {
#pragma unroll
                  for (int i = 0; i < kVec; ++i)
                    if (i < nelem - e0) E::store1(o + i * E::kBytes, d[i]);
                }
              }
            }
          }
          if (c == p.cy) {
            // the owner of the sampled id rewrites its vector with the -g term
            // (after its own store of that vector, so program order settles it)
            float d[kVec];
            const uint4 w = ld_shared_v4(buf + p.jv / kVec * 16);
            grad_vec<E, kEnt>(w, cf.cL, cf.cL_lo, cf.a0, cf.a1, d);
#pragma unroll
            for (int i = 0; i < kVec; ++i)
              if (i == p.jv % kVec) d[i] -= cf.gy;
            const int e0 = c0 + p.jv / kVec * kVec;
            unsigned char* o = drow + static_cast<long long>(e0) * E::kBytes;
            if (nelem - e0 >= kVec) {
              st_global_cs_v4(o, E::pack(d));
            } else {
#pragma unroll
              for (int i = 0; i < kVec; ++i)
                if (i < nelem - e0) E::store1(o + i * E::kBytes, d[i]);
            }
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_addr(&sm.empty[slot]));
      }
    };

    // the rows of this CTA; the id of the row after the current one is loaded a row ahead
    RowWalk<true> walk(cid, ncl);
    long long cur = walk.next(a.mask, ncl, a.R, lane);
    long long nxt = walk.next(a.mask, ncl, a.R, lane);
    IdPos pc = id_pos<kChunkElems, kVec>(a, cur < a.R ? a.ids[cur] : 0, tid);
    long long y_nxt = nxt < a.R ? a.ids[nxt] : 0;
    auto advance = [&]() {
      cur = nxt;
      pc = id_pos<kChunkElems, kVec>(a, y_nxt, tid);
      nxt = walk.next(a.mask, ncl, a.R, lane);
      y_nxt = nxt < a.R ? a.ids[nxt] : 0;
    };
    uint32_t k = 0;
    if constexpr (kMode == 0) {
      // Each step: the first `lead` chunks of the current row's pass 1, pass 2
      // of the previous row, then the rest of the current row's pass 1 (the
      // first step has no previous row, the last no current one).  One copy
      // of each pass's code in the loop keeps the kernel's instruction
      // footprint small.
      long long prev = -1;
      IdPos pp = pc;
      uint32_t kp = 0, base_p = 0;
      while ((cur < a.R || prev >= 0) && (kMeet || !*abort_flag)) {
        const bool has_cur = cur < a.R;
        if (RL_ZERO_WARP && tid == 0 && has_cur) *reinterpret_cast<volatile long long*>(&sm.pace) = cur;
        const int lead = !has_cur ? 0 : prev >= 0 ? min(nchunks, lead_chunks) : nchunks;
        const uint32_t base = it;  // resident rows: ring position of the current row's first chunk
        ThreadStats st;
        stats_init(st);
        float zy = -INFINITY, m0 = kFloor, s0 = 0.f, t0 = 0.f;
#pragma unroll 1
        for (int seg = 0; seg < 2; ++seg) {
          const int c0 = seg == 0 ? 0 : lead;
          const int c1 = !has_cur ? 0 : seg == 0 ? lead : nchunks;
          pass1(c0, c1, st, zy, pc);
          if (seg == 0) {
            if (lead > 0) {  // the current row's first chunks, kept as one (m, s, t) over pass 2
              fold(st, m0, s0, t0);
              stats_init(st);
            }
            if (prev >= 0) pass2(prev, kp, base_p, pp);
          }
        }
        if (has_cur) publish(k, st, m0, s0, t0, zy, pc);
        prev = has_cur ? cur : -1;
        pp = pc;
        kp = k;
        base_p = base;
        if (has_cur) {
          advance();
          ++k;
        }
      }
    } else {
      for (; cur < a.R && (kMeet || !*abort_flag); ++k) {
        if (RL_ZERO_WARP && tid == 0) *reinterpret_cast<volatile long long*>(&sm.pace) = cur;
        if constexpr (kMode == 1) {
          ThreadStats st;
          stats_init(st);
          float zy = -INFINITY;
          pass1(0, nchunks, st, zy, pc);
          publish(k, st, kFloor, 0.f, 0.f, zy, pc);
        } else {
          pass2(cur, k, 0, pc);
        }
        advance();
      }
    }
    if (RL_ZERO_WARP && tid == 0) *reinterpret_cast<volatile long long*>(&sm.pace) = a.R + 1;  // release the zero warp
  }

  // ---- per-CTA partial (the warps' sums in warp order), then the last CTA
  //      reduces all partials in CTA order
  if (lane == 0) {
    for (int q = 0; q < 5; ++q) sm.wred[warp][q] = wacc[q];
    if (err) atomicOr(&a.ws->status, err);
  }
  named_barrier(kRedBarrier, kRedThreads);
  if (tid == 0) {
    WsPartial& P = a.partials[blockIdx.x];
    for (int q = 0; q < 5; ++q) {
      double v = 0.0;
      for (int w = 0; w < kRedWarps; ++w) v += sm.wred[w][q];
      P.v[q] = v;
    }
    if (*abort_flag) atomicOr(&a.ws->status, static_cast<unsigned int>(RL_DEVERR_TIMEOUT));
    __threadfence();
    const unsigned int ticket = atomicInc(&a.ws->ticket, gridDim.x - 1);
    sm.is_last = (ticket == gridDim.x - 1);
  }
  named_barrier(kRedBarrier, kRedThreads);
  if (sm.is_last) {
    __threadfence();
    double v[5] = {0.0, 0.0, 0.0, 0.0, 0.0};
    for (int i = tid; i < static_cast<int>(gridDim.x); i += kRedThreads)
      for (int q = 0; q < 5; ++q) v[q] += __ldcg(&a.partials[i].v[q]);
    for (int q = 0; q < 5; ++q) v[q] = warp_sum_d(v[q]);
    if (lane == 0)
      for (int q = 0; q < 5; ++q) sm.wred[warp][q] = v[q];
    named_barrier(kRedBarrier, kRedThreads);
    if (tid == 0) {
      double tot[5] = {0.0, 0.0, 0.0, 0.0, 0.0};
      for (int w = 0; w < kRedWarps; ++w)
        for (int q = 0; q < 5; ++q) tot[q] += sm.wred[w][q];
      const unsigned int stw = atomicExch(&a.ws->status, 0u);
      a.ws->last_status = stw;
      rl_loss_stats out;
      const double inv = N > 0 ? 1.0 / static_cast<double>(N) : 0.0;
      out.loss = a.agg == RL_AGG_TOKEN_MEAN ? -tot[0] * inv : (N > 0 ? -tot[0] : 0.0);
      out.pg_term = tot[1] * inv;
      out.kl_term = tot[2] * inv;
      out.ent_term = tot[3] * inv;
      out.clip_frac = tot[4] * inv;
      out.n_tokens = N_local;
      out.n_clipped = static_cast<long long>(tot[4]);
      out.device_error = static_cast<int>(stw);
      out.reserved = 0;
      *a.stats = out;
    }
  }
}

// ------------------------------------------------------------------ host side
int elem_bytes(rl_dtype dt) {
  switch (dt) {
    case RL_F32: return 4;
    case RL_BF16: return 2;
    case RL_F16: return 2;
  }
  return 0;
}

struct Plan {
  int cluster;      // CTAs per row (always 1; the launch shape reports it)
  int n_clusters;   // CTAs (rows in flight) in the persistent grid
  bool stream;      // rows streamed twice (second pass from L2)
};

// Row layout: a row that fits the ring twice over stays in shared memory for
// both passes; a longer one is streamed.
bool choose_layout(int es, long long V, Plan* p) {
  if (V > (1LL << 30)) return false;  // element offsets within a row are 32-bit
  const long long row_chunks = ((V * es + 15) / 16 * 16 + kChunkBytes - 1) / kChunkBytes;
  p->cluster = 1;
  p->stream = row_chunks > kMaxResidentChunks;
  return true;
}

// The entropy term is a template argument (c_ent != 0); the statistics-only
// mode has no gradient and is built without it.
template <int DT, int M, bool E>
void* kernel_ptr(bool stream) {
  return stream ? reinterpret_cast<void*>(&RL_LOSS_KERNEL<DT, true, M, E>)
                : reinterpret_cast<void*>(&RL_LOSS_KERNEL<DT, false, M, E>);
}

template <int M, bool E>
void* kernel_for_mode(rl_dtype dt, bool stream) {
  switch (dt) {
    case RL_F32: return kernel_ptr<RL_F32, M, E>(stream);
    case RL_BF16: return kernel_ptr<RL_BF16, M, E>(stream);
    case RL_F16: return kernel_ptr<RL_F16, M, E>(stream);
  }
  return nullptr;
}

void* kernel_for(rl_dtype dt, bool stream, int mode, bool ent) {
  // no columns: the element format and row layout do not matter
  if (mode == 3) return reinterpret_cast<void*>(&RL_LOSS_KERNEL<RL_BF16, false, 3, false>);
  if (mode == 1) return kernel_for_mode<1, false>(dt, stream);
  if (mode == 2) return ent ? kernel_for_mode<2, true>(dt, stream) : kernel_for_mode<2, false>(dt, stream);
  return ent ? kernel_for_mode<0, true>(dt, stream) : kernel_for_mode<0, false>(dt, stream);
}

// Per (device, kernel, cluster size): attributes set once and the number of
// co-resident clusters.
std::mutex g_occ_mu;
std::map<std::tuple<int, int, int, int, int>, int> g_occ;

rl_status max_clusters(rl_dtype dt, bool stream, int cluster, int mode, int* out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return RL_ERR_CUDA;
  const auto key = std::make_tuple(dev, static_cast<int>(dt), static_cast<int>(stream), cluster, mode);
  std::lock_guard<std::mutex> lock(g_occ_mu);
  auto found = g_occ.find(key);
  if (found != g_occ.end()) {
    *out = found->second;
    return RL_OK;
  }
  // both entropy variants get the shared-memory attribute; they have the same occupancy
  void* fn = kernel_for(dt, stream, mode, false);
  void* fn_ent = kernel_for(dt, stream, mode, true);
  const int smem = static_cast<int>(sizeof(LossSmem));
  if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess ||
      cudaFuncSetAttribute(fn_ent, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
    return RL_ERR_CUDA;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(cluster);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, fn, &cfg) != cudaSuccess || n < 1) return RL_ERR_CUDA;
  g_occ[key] = n;
  *out = n;
  return RL_OK;
}

rl_status plan(rl_dtype dt, long long V, long long R, Plan* p, int mode = 0) {
  const int es = elem_bytes(dt);
  if (es == 0) return RL_ERR_DTYPE;
  if (V < (mode >= 2 ? 0 : 1) || R < 0) return RL_ERR_SHAPE;
  if (!choose_layout(es, V, p)) return RL_ERR_SHAPE;
  int occ = 0;
  const rl_status st = max_clusters(dt, p->stream, p->cluster, mode, &occ);
  if (st != RL_OK) return st;
  long long n = occ;
  if (n > R) n = R > 0 ? R : 1;
  if (n * p->cluster > kMaxGrid) n = kMaxGrid / p->cluster;
  p->n_clusters = static_cast<int>(n);
  return RL_OK;
}

bool finite(float x) { return std::isfinite(x); }

}  // namespace
}  // namespace rl

using namespace rl;

// ------------------------------------------------------------------ launch
namespace {
template <int DT, bool S>
cudaError_t launch_one(cudaLaunchConfig_t* cfg, int mode, bool ent, const LossArgs& args) {
  if (mode == 3) return cudaLaunchKernelEx(cfg, RL_LOSS_KERNEL<RL_BF16, false, 3, false>, args);
  if (mode == 1) return cudaLaunchKernelEx(cfg, RL_LOSS_KERNEL<DT, S, 1, false>, args);
  if (mode == 2)
    return ent ? cudaLaunchKernelEx(cfg, RL_LOSS_KERNEL<DT, S, 2, true>, args)
               : cudaLaunchKernelEx(cfg, RL_LOSS_KERNEL<DT, S, 2, false>, args);
  return ent ? cudaLaunchKernelEx(cfg, RL_LOSS_KERNEL<DT, S, 0, true>, args)
             : cudaLaunchKernelEx(cfg, RL_LOSS_KERNEL<DT, S, 0, false>, args);
}

template <int DT>
cudaError_t launch_mode(cudaLaunchConfig_t* cfg, bool stream, int mode, bool ent, const LossArgs& args) {
  return stream ? launch_one<DT, true>(cfg, mode, ent, args) : launch_one<DT, false>(cfg, mode, ent, args);
}
}  // namespace

// ------------------------------------------------------------------ this build's entry
namespace RL_ROWS_NS {

RL_INTERNAL rl_status launch_shape(rl_dtype dtype, long long V, long long n_rows, int* cluster_size,
                                   int* n_clusters, int* smem_bytes) {
  Plan p;
  const rl_status st = plan(dtype, V, n_rows, &p);
  if (st != RL_OK) return st;
  *cluster_size = p.cluster;
  *n_clusters = p.n_clusters;
  *smem_bytes = static_cast<int>(sizeof(LossSmem));
  return RL_OK;
}

RL_INTERNAL rl_status fwd_bwd(const rl_policy_loss_desc* d, void* stream) {
  const int es = elem_bytes(d->dtype);
  if (es == 0) return RL_ERR_DTYPE;
  if (d->adv_layout != RL_ADV_PER_SEQ && d->adv_layout != RL_ADV_PER_TOKEN &&
      d->adv_layout != RL_ADV_GROUP_REWARDS)
    return RL_ERR_DTYPE;
  if (d->agg != RL_AGG_TOKEN_MEAN && d->agg != RL_AGG_SEQ_MEAN_TOKEN_MEAN &&
      d->agg != RL_AGG_SEQ_MEAN_TOKEN_SUM && d->agg != RL_AGG_TOKEN_SUM_NORM)
    return RL_ERR_DTYPE;
  const long long B = d->B, T = d->T, V = d->V, ld = d->ld;
  // A merge launch that only writes row coefficients may have no columns of its own.
  const bool coef_only = d->shard_partials && d->row_coef_out && V == 0;
  if (coef_only && d->vocab_total < 1) return RL_ERR_SHAPE;
  if (B < 0 || T < 0 || V < (coef_only ? 0 : 1) || ld < V) return RL_ERR_SHAPE;
  if (B > 0 && T > (1LL << 40) / B) return RL_ERR_SHAPE;
  const long long R = B * T;
  if (!d->stats_dev) return RL_ERR_NULL;
  if (!d->workspace || d->workspace_bytes < kWorkspaceBytes) return RL_ERR_WORKSPACE;
  if (R > 0 && ((!d->logits && !coef_only) || !d->ids || !d->mask || !d->adv)) return RL_ERR_NULL;
  if (d->row_coef_out && !d->shard_partials) return RL_ERR_ARG;
  if ((reinterpret_cast<uintptr_t>(d->row_coef_out) & 15) != 0) return RL_ERR_ALIGN;
  if (d->beta != 0.f && !d->ref_logp) return RL_ERR_NULL;
  if (!finite(d->eps) || d->eps < 0.f || !finite(d->eps_high) || !finite(d->beta) ||
      !finite(d->c_ent) || !finite(d->grad_scale))
    return RL_ERR_ARG;
  if (d->adv_layout == RL_ADV_GROUP_REWARDS) {
    if (d->ddof != 0 && d->ddof != 1) return RL_ERR_ARG;
    if (!(d->std_eps >= 0.0) || !std::isfinite(d->std_eps)) return RL_ERR_ARG;
    if (d->group_size <= d->ddof || d->group_size < 1 || B % d->group_size != 0) return RL_ERR_SHAPE;
  }
  if (d->agg == RL_AGG_TOKEN_SUM_NORM && !(d->agg_norm > 0.0 && std::isfinite(d->agg_norm)))
    return RL_ERR_ARG;
  // vocabulary shards; a merge launch with no columns of its own runs warp-parallel rows
  const int mode = d->partials_out ? 1 : d->shard_partials ? (coef_only ? 3 : 2) : 0;
  const long long v_total = d->vocab_total > 0 ? d->vocab_total : V;
  if (d->partials_out && d->shard_partials) return RL_ERR_ARG;
  if (d->vocab_offset < 0 || d->vocab_total < 0 || d->vocab_offset + V > v_total) return RL_ERR_SHAPE;
  if (mode >= 2 && d->n_shards < 1) return RL_ERR_ARG;
  if ((reinterpret_cast<uintptr_t>(d->partials_out) & 15) != 0 ||
      (reinterpret_cast<uintptr_t>(d->shard_partials) & 15) != 0)
    return RL_ERR_ALIGN;
  const long long row_bytes = ld * es;
  if ((row_bytes & 15) != 0) return RL_ERR_ALIGN;
  if ((reinterpret_cast<uintptr_t>(d->logits) & 15) != 0) return RL_ERR_ALIGN;
  if ((reinterpret_cast<uintptr_t>(d->dlogits) & 15) != 0) return RL_ERR_ALIGN;
  if ((reinterpret_cast<uintptr_t>(d->workspace) & 15) != 0) return RL_ERR_ALIGN;
  if (d->dlogits && d->dlogits != d->logits && R > 0) {
    const uintptr_t l0 = reinterpret_cast<uintptr_t>(d->logits);
    const uintptr_t d0 = reinterpret_cast<uintptr_t>(d->dlogits);
    const uintptr_t n = static_cast<uintptr_t>(R) * static_cast<uintptr_t>(row_bytes);
    if (l0 < d0 + n && d0 < l0 + n) return RL_ERR_ALIAS;
  }

  Plan pl;
  const rl_status st = plan(d->dtype, V, R, &pl, mode);
  if (st != RL_OK) return st;

  LossArgs args;
  args.logits = static_cast<const unsigned char*>(d->logits);
  args.dlogits = static_cast<unsigned char*>(d->dlogits);
  args.ids = d->ids;
  args.logp_old = d->logp_old;
  args.ref_logp = d->ref_logp;
  args.mask = d->mask;
  args.adv = d->adv;
  args.logp_out = d->logp_out;
  args.entropy_out = d->entropy_out;
  args.stats = d->stats_dev;
  args.ws = static_cast<WsHeader*>(d->workspace);
  args.partials =
      reinterpret_cast<WsPartial*>(static_cast<unsigned char*>(d->workspace) + sizeof(WsHeader));
  args.R = R;
  args.T = T > 0 ? T : 1;
  args.V = V;
  args.row_bytes = row_bytes;
  args.adv_mode = d->adv_layout;
  args.group_size = d->group_size;
  args.ddof = d->ddof;
  args.std_eps = d->std_eps;
  args.clip_lo = 1.f - d->eps;
  args.clip_hi = 1.f + (d->eps_high < 0.f ? d->eps : d->eps_high);
  args.beta = d->beta;
  args.c_ent = d->c_ent;
  args.grad_scale = d->grad_scale;
  args.agg = d->agg;
  args.agg_w = d->agg == RL_AGG_TOKEN_SUM_NORM ? 1.0 / d->agg_norm : 0.0;
  args.global_counts = d->global_counts;
  args.v_offset = d->vocab_offset;
  args.v_total = v_total;
  args.partials_out = reinterpret_cast<float4*>(d->partials_out);
  args.shard_partials = reinterpret_cast<const float4*>(d->shard_partials);
  args.n_shards = mode >= 2 ? d->n_shards : 0;
  args.row_coef_out = reinterpret_cast<float4*>(d->row_coef_out);
  if (coef_only) args.dlogits = nullptr;
  if (mode == 1) {  // statistics only
    args.dlogits = nullptr;
    args.logp_out = nullptr;
    args.entropy_out = nullptr;
  }

  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = pl.cluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3(static_cast<unsigned>(pl.cluster * pl.n_clusters));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = sizeof(LossSmem);
  cfg.stream = static_cast<cudaStream_t>(stream);
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  cudaError_t e = cudaErrorInvalidValue;
  switch (d->dtype) {
    case RL_F32: e = launch_mode<RL_F32>(&cfg, pl.stream, mode, d->c_ent != 0.f, args); break;
    case RL_BF16: e = launch_mode<RL_BF16>(&cfg, pl.stream, mode, d->c_ent != 0.f, args); break;
    case RL_F16: e = launch_mode<RL_F16>(&cfg, pl.stream, mode, d->c_ent != 0.f, args); break;
  }
  return e == cudaSuccess ? RL_OK : RL_ERR_CUDA;
}

}  // namespace RL_ROWS_NS

#ifndef RL_SHORT_ROWS
// ------------------------------------------------------------------ C entry points
namespace rl_short_rows {
RL_INTERNAL rl_status launch_shape(rl_dtype dtype, long long V, long long n_rows, int* cluster_size,
                                   int* n_clusters, int* smem_bytes);
RL_INTERNAL rl_status fwd_bwd(const rl_policy_loss_desc* d, void* stream);
}  // namespace rl_short_rows

namespace {
// Rows (this call's columns) of at most this many bytes take the short-row
// build: two CTAs per SM measured faster up to 100 KB rows (V = 50,000
// bf16) and slower from 128 KB on when most rows are masked.
#ifndef RL_SHORT_ROW_BYTES
#define RL_SHORT_ROW_BYTES 102400
#endif
constexpr long long kShortRowBytes = RL_SHORT_ROW_BYTES;

bool short_rows(rl_dtype dtype, long long V) {
  const int es = elem_bytes(dtype);
  return es > 0 && V >= 1 && V <= kShortRowBytes / es;
}
}  // namespace

// Scratch for rl_policy_loss_fwd_bwd_noalloc: the workspace a caller would
// otherwise allocate (status header + one partial per CTA, kWorkspaceBytes =
// 131,328 bytes), held in a file-scope device array instead.  Every GPU that
// loads the library holds it until the process exits.  plan() never gives a
// grid of more than kMaxGrid CTAs, so the array covers every call.
static __device__ __align__(256) unsigned char g_loss_scratch[kWorkspaceBytes];
static_assert(sizeof(g_loss_scratch) >= sizeof(WsHeader) + sizeof(WsPartial) * kMaxGrid,
              "the static scratch holds the workspace of the largest grid plan() gives");

namespace {
// In host code g_loss_scratch names a host-side stand-in, not device memory:
// the device address comes from cudaGetSymbolAddress with the target device
// current.  It is looked up on every call rather than cached, so that a
// cudaDeviceReset, or another context made current on the same device, never
// leaves a stale address behind (the lookup is a host-side table read once
// the module is loaded; the first call on a device loads it).
rl_status loss_scratch_address(void** out) {
  void* ptr = nullptr;
  if (cudaGetSymbolAddress(&ptr, g_loss_scratch) != cudaSuccess || ptr == nullptr)
    return RL_ERR_CUDA;
  *out = ptr;
  return RL_OK;
}
}  // namespace

extern "C" size_t rl_policy_loss_workspace_size(long long n_rows) {
  (void)n_rows;
  return kWorkspaceBytes;
}

extern "C" rl_status rl_policy_loss_launch_shape(rl_dtype dtype, long long V, long long n_rows,
                                                 int* cluster_size, int* n_clusters,
                                                 int* smem_bytes) {
  if (!cluster_size || !n_clusters || !smem_bytes) return RL_ERR_NULL;
  return short_rows(dtype, V) ? rl_short_rows::launch_shape(dtype, V, n_rows, cluster_size, n_clusters, smem_bytes)
                              : rl_long_rows::launch_shape(dtype, V, n_rows, cluster_size, n_clusters, smem_bytes);
}

extern "C" void rl_policy_loss_desc_init(rl_policy_loss_desc* d) {
  if (!d) return;
  std::memset(d, 0, sizeof(*d));
  d->dtype = RL_BF16;
  d->adv_layout = RL_ADV_PER_SEQ;
  d->group_size = 1;
  d->ddof = 1;
  d->std_eps = 1e-4;
  d->eps = 0.2f;
  d->eps_high = -1.f;
  d->grad_scale = 1.f;
  d->agg = RL_AGG_TOKEN_MEAN;
  d->agg_norm = 1.0;
}

extern "C" rl_status rl_policy_loss_fwd_bwd_ex(const rl_policy_loss_desc* d, void* stream) {
  if (!d) return RL_ERR_NULL;
  return short_rows(d->dtype, d->V) ? rl_short_rows::fwd_bwd(d, stream) : rl_long_rows::fwd_bwd(d, stream);
}

extern "C" rl_status rl_policy_loss_fwd_bwd(const void* logits, rl_dtype dtype, long long B,
                                            long long T, long long V, long long ld,
                                            const long long* ids, const float* logp_old,
                                            const float* ref_logp, const unsigned char* mask,
                                            const float* adv, rl_adv_layout adv_layout, float eps,
                                            float beta, float c_ent, float grad_scale,
                                            void* dlogits, float* logp_out, float* entropy_out,
                                            rl_loss_stats* stats_dev, void* workspace,
                                            size_t workspace_bytes, void* stream) {
  // The fixed-argument form covers given advantages only.
  if (adv_layout != RL_ADV_PER_SEQ && adv_layout != RL_ADV_PER_TOKEN) return RL_ERR_DTYPE;
  rl_policy_loss_desc d;
  rl_policy_loss_desc_init(&d);
  d.logits = logits;
  d.dtype = dtype;
  d.B = B;
  d.T = T;
  d.V = V;
  d.ld = ld;
  d.ids = ids;
  d.logp_old = logp_old;
  d.ref_logp = ref_logp;
  d.mask = mask;
  d.adv = adv;
  d.adv_layout = adv_layout;
  d.eps = eps;
  d.eps_high = eps;
  d.beta = beta;
  d.c_ent = c_ent;
  d.grad_scale = grad_scale;
  d.dlogits = dlogits;
  d.logp_out = logp_out;
  d.entropy_out = entropy_out;
  d.stats_dev = stats_dev;
  d.workspace = workspace;
  d.workspace_bytes = workspace_bytes;
  return rl_policy_loss_fwd_bwd_ex(&d, stream);
}

extern "C" rl_status rl_policy_loss_fwd_bwd_noalloc(
    const void* logits, rl_dtype dtype, long long B, long long T, long long V, long long ld,
    const long long* ids, const float* logp_old, const float* ref_logp, const unsigned char* mask,
    const float* adv, rl_adv_layout adv_layout, float eps, float beta, float c_ent,
    float grad_scale, void* dlogits, float* logp_out, float* entropy_out,
    rl_loss_stats* stats_dev, void* stream) {
  if (B < 0 || T < 0) return RL_ERR_SHAPE;
  if (B > 0 && T > (1LL << 40) / B) return RL_ERR_SHAPE;
  // The scratch this call's grid needs: the header and one partial per CTA.
  int cluster = 0, n_clusters = 0, smem = 0;
  const rl_status shape = rl_policy_loss_launch_shape(dtype, V, B * T, &cluster, &n_clusters, &smem);
  if (shape != RL_OK) return shape;
  if (sizeof(WsHeader) + sizeof(WsPartial) * static_cast<size_t>(cluster) * n_clusters > sizeof(g_loss_scratch))
    return RL_ERR_WORKSPACE;
  void* scratch = nullptr;
  const rl_status st = loss_scratch_address(&scratch);
  if (st != RL_OK) return st;
  // The status word and the last-CTA ticket must start at zero; the array
  // keeps whatever the previous call left, so clear the header on the stream.
  if (cudaMemsetAsync(scratch, 0, sizeof(WsHeader), static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return RL_ERR_CUDA;
  return rl_policy_loss_fwd_bwd(logits, dtype, B, T, V, ld, ids, logp_old, ref_logp, mask, adv,
                                adv_layout, eps, beta, c_ent, grad_scale, dlogits, logp_out,
                                entropy_out, stats_dev, scratch, sizeof(g_loss_scratch), stream);
}
#endif  // !RL_SHORT_ROWS
