/*
 * rlloss.h — C ABI of the fused RL policy-loss library (GB300, sm_103a).
 *
 * The library computes the data-parallel hot path of an LLM reinforcement-
 * learning update: reward normalisation into advantages, then, in ONE kernel
 * launch, the per-token log-softmax over the vocabulary, the clipped
 * surrogate objective with a KL penalty and an entropy bonus, the masked-mean
 * loss and the gradient of that loss with respect to the logits.
 *
 * Sources (RL.cu, "LLM Reinforcement Learning in Pure CUDA"):
 *   - ainews.cool RL.cu article, section "技术深度解析" (technical deep dive),
 *     bullet "PPO 更新内核" (PPO update kernel): advantage estimation, clipped
 *     surrogate objective and entropy bonus fused into a single kernel launch
 *     to cut global-memory round trips; bullet "滚动缓冲区" (rollout buffer):
 *     a fixed-size, preallocated GPU buffer of states, actions, rewards and
 *     log-probabilities, memory managed by the caller;
 *   - the same article, paragraph after its benchmark table: KL-divergence
 *     penalty and reward normalisation, and CUDA-graph capture of the whole
 *     training step;
 *   - pitchhut.com RL.cu listing, "Key Features" item 3 and mlllm.io RL.cu
 *     article, "Что произошло": the method is GRPO (group-relative policy
 *     optimisation), i.e. group-normalised rewards as advantages;
 *   - pitchhut.com RL.cu listing, "Key Features" item 1: FP16 inputs with FP32
 *     accumulation.
 * The pages print no formula; each entry point below states the standard
 * definition it computes.
 *
 * Conventions for every entry point:
 *   - Every array pointer is DEVICE memory owned by the caller.  The library
 *     never allocates or frees memory and keeps no per-call host state.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Calls are asynchronous and stream-ordered; none synchronises
 *     except rl_read_device_status.
 *   - Argument errors are detected on the host before anything is launched
 *     and returned synchronously; nothing is written in that case.  A launch
 *     failure returns RL_ERR_CUDA.
 *   - Device-detected errors never trap: they set bits in the call's status
 *     (rl_loss_stats.device_error and the workspace status word), the
 *     affected outputs become NaN, and the kernel returns normally.
 */
#ifndef RLLOSS_H
#define RLLOSS_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  RL_OK = 0,
  RL_ERR_NULL = 1,       /* a required pointer is NULL */
  RL_ERR_SHAPE = 2,      /* a size is negative, zero where it must not be, or too large */
  RL_ERR_DTYPE = 3,      /* unknown element type or advantage layout */
  RL_ERR_ALIGN = 4,      /* a logits/dlogits base or row stride is not 16-byte aligned */
  RL_ERR_ALIAS = 5,      /* dlogits partially overlaps logits */
  RL_ERR_WORKSPACE = 6,  /* workspace NULL or smaller than rl_policy_loss_workspace_size() */
  RL_ERR_ID_RANGE = 7,   /* (device) a sampled id outside [0, V) on a valid token */
  RL_ERR_TIMEOUT = 8,    /* (device) a bounded on-chip wait gave up; outputs are garbage */
  RL_ERR_CUDA = 9,       /* a CUDA runtime call or launch failed */
  RL_ERR_ARG = 10        /* a scalar argument is out of range (NaN, negative eps, ...) */
} rl_status;

typedef enum { RL_F32 = 0, RL_BF16 = 1, RL_F16 = 2 } rl_dtype;

typedef enum {
  RL_ADV_PER_SEQ = 0,      /* adv[B]: one advantage per sequence (GRPO) */
  RL_ADV_PER_TOKEN = 1,    /* adv[B*T]: one advantage per token (PPO-GAE) */
  RL_ADV_GROUP_REWARDS = 2 /* adv[B] holds the sequences' REWARDS; the loss launch
                              computes the group-relative advantages itself
                              (rl_policy_loss_fwd_bwd_ex only) */
} rl_adv_layout;

/* How token objectives are averaged into the loss (loss = -sum_t w_t J_t). */
typedef enum {
  RL_AGG_TOKEN_MEAN = 0,          /* w = 1/N: one mean over all valid tokens */
  RL_AGG_SEQ_MEAN_TOKEN_MEAN = 1, /* w = 1/(B' L_b): mean over sequences of their token means */
  RL_AGG_SEQ_MEAN_TOKEN_SUM = 2,  /* w = 1/B': mean over sequences of their token sums */
  RL_AGG_TOKEN_SUM_NORM = 3       /* w = 1/agg_norm: token sum over a fixed normaliser */
} rl_loss_agg;

/* Device-error bits of rl_loss_stats.device_error and of the workspace word. */
#define RL_DEVERR_ID_RANGE 1u
#define RL_DEVERR_TIMEOUT 2u

/*
 * Scalar results of one rl_policy_loss_fwd_bwd call, written by the kernel
 * into caller-owned device memory.  All means are over the N valid tokens
 * (N = 0 gives all zeros).
 *   loss      = -(1/N) sum_t m_t J_t
 *   pg_term   =  (1/N) sum_t m_t pg_t       (clipped surrogate)
 *   kl_term   =  (1/N) sum_t m_t kl_t       (k3 estimator)
 *   ent_term  =  (1/N) sum_t m_t H_t        (entropy)
 *   clip_frac = n_clipped / N, n_clipped = tokens whose surrogate gradient is
 *               cut by the clip: (A > 0 and r > 1+eps) or (A < 0 and r < 1-eps)
 */
typedef struct {
  double loss;
  double pg_term;
  double kl_term;
  double ent_term;
  double clip_frac;
  long long n_tokens;
  long long n_clipped;
  int device_error;      /* RL_DEVERR_* bits seen during this call */
  int reserved;
} rl_loss_stats;

/*
 * Group-relative advantages (GRPO reward normalisation).
 *   For group g with rewards R_{g,0..G-1} (sequence i = g*G + j, group-major):
 *     mean = (1/G) sum_j R_j,  std = sqrt( sum_j (R_j - mean)^2 / (G - ddof) )
 *     adv_out[i] = (R_i - mean) / (std + std_eps)
 *   rewards  : float[n_groups * group_size], device, read only.
 *   adv_out  : float[n_groups * group_size], device, written (may equal rewards).
 *   std_eps  : the stabiliser added to std (1e-4 in the usual GRPO recipe).
 *   ddof     : 1 (unbiased, default reading) or 0.
 * Arithmetic in fp64, result rounded to fp32.  One launch, one warp per group.
 * Errors: RL_ERR_NULL, RL_ERR_SHAPE (n_groups < 0, group_size < 1,
 * group_size <= ddof), RL_ERR_ARG (ddof not 0/1, std_eps negative or NaN).
 * n_groups == 0 launches nothing and returns RL_OK.
 */
rl_status rl_group_advantages(const float* rewards, int n_groups, int group_size,
                              double std_eps, int ddof, float* adv_out, void* stream);

/*
 * PPO generalised advantage estimation, reverse scan over time.
 *   For sequence b with length L = clamp(lengths[b], 0, T), t = L-1 .. 0:
 *     delta_t = r_t + gamma * (t+1 < L ? v_{t+1} : 0) - v_t
 *     A_t     = delta_t + gamma * lam * (t+1 < L ? A_{t+1} : 0)
 *     ret_t   = A_t + v_t
 *   and A_t = ret_t = 0 for t >= L (the episode ends at L-1; bootstrap 0).
 *   rewards, values : float[B*T] row-major [B, T], device, read only.
 *   lengths         : int[B], device (values outside [0, T] are clamped).
 *   adv_out         : float[B*T], device, written.
 *   returns_out     : float[B*T], device, written; may be NULL.
 * Arithmetic in fp64 (a warp-parallel affine scan over the sequence),
 * result rounded to fp32.  One launch, one CTA per sequence.
 * Errors: RL_ERR_NULL, RL_ERR_SHAPE (B < 0, T < 0), RL_ERR_ARG (NaN gamma/lam).
 */
rl_status rl_gae_reverse_scan(const float* rewards, const float* values, const int* lengths,
                              int B, int T, float gamma, float lam,
                              float* adv_out, float* returns_out, void* stream);

/*
 * Masked advantage whitening over the valid tokens of the batch (the usual
 * normalisation of PPO-GAE advantages; the pages name reward normalisation and
 * advantage estimation in the update, ainews.cool RL.cu article):
 *   mu = (1/N) sum_t m_t x_t,  var = (1/(N-1)) sum_t m_t (x_t - mu)^2  (0 if N < 2)
 *   out_t = (x_t - mu) / sqrt(var + eps)   (x_t / sqrt(var + eps) if !shift_mean)
 *   out_t = 0 where mask_t == 0.
 *   x, out : float[n], device (out may equal x);  mask : uint8[n].
 * fp32 per element, fp64 reductions in a fixed order, one launch of one
 * CTA.  Errors: RL_ERR_SHAPE (n < 0), RL_ERR_NULL, RL_ERR_ARG (eps negative
 * or NaN).  n == 0 launches nothing.
 */
rl_status rl_masked_whiten(const float* x, const unsigned char* mask, long long n, double eps,
                           int shift_mean, float* out, void* stream);

/*
 * Bytes of device workspace rl_policy_loss_fwd_bwd needs for n_rows rows.
 * The workspace must be zero-filled once before its first use (e.g. with
 * cudaMemset); every call that completes leaves it ready for the next.  A
 * workspace serves one call at a time: two calls in flight on it race.
 */
size_t rl_policy_loss_workspace_size(long long n_rows);

/*
 * The fused policy-loss forward and backward, in one kernel launch.
 *
 * Rows: row = b*T + t for sequence b, position t; R = B*T rows of V logits.
 * For every row with mask[row] != 0 (a valid token; N = number of them):
 *   z = logits row, y = ids[row]
 *   lse = log sum_v exp(z_v),  logp = z_y - lse,  p_v = exp(z_v - lse)
 *   H   = -sum_v p_v log p_v                                  (entropy)
 *   r   = exp(logp - logp_old[row])            (r = 1 if logp_old == NULL)
 *   A   = adv[b] (RL_ADV_PER_SEQ) or adv[row] (RL_ADV_PER_TOKEN)
 *   pg  = min(r A, clamp(r, 1-eps, 1+eps) A)                  (clipped surrogate)
 *   d   = ref_logp[row] - logp,  kl = exp(d) - d - 1          (k3; 0 if beta == 0
 *                                                              and ref_logp == NULL)
 *   J   = pg - beta kl + c_ent H
 * loss = -(1/N) sum_rows J.  The gradient written to dlogits is
 *   dz_v = grad_scale (1/N) [ g (p_v - [v == y]) + c_ent p_v (log p_v + H) ]
 *   g    = pg' + beta (exp(d) - 1),  pg' = r A unless (A > 0 and r > 1+eps) or
 *          (A < 0 and r < 1-eps), where pg' = 0 (the clip is inclusive at 1+-eps).
 * Rows with mask 0 get an all-zero dlogits row, logp_out = entropy_out = 0,
 * and neither their logits nor their id is read.  N = 0 gives loss 0 and an
 * all-zero gradient.
 *
 * Arguments:
 *   logits      : [R, ld] elements of `dtype`, row-major, device, read only.
 *                 Base address 16-byte aligned; ld * sizeof(dtype) a multiple
 *                 of 16 (pad rows if V is odd); ld >= V.
 *   dtype       : RL_F32, RL_BF16 or RL_F16 (for logits and dlogits alike).
 *   B, T, V, ld : B >= 0, T >= 0, 1 <= V <= 2^30.  A row that fits two
 *                 chunks of the kernel's shared-memory ring stays on chip for
 *                 both passes: rows of at most 32 KB (short-row build, 16 KB
 *                 chunks, rows up to 100 KB) or 64 KB (long-row build, 32 KB
 *                 chunks, rows over 100 KB).  Other rows are streamed through
 *                 shared memory twice, the second time from L2 (a 64 KB row,
 *                 e.g. V = 32000 fp16, takes the short-row build and is
 *                 streamed).  Larger V returns RL_ERR_SHAPE.
 *   ids         : int64[R], the sampled token of each row.  An id outside
 *                 [0, V) on a valid row sets RL_DEVERR_ID_RANGE and makes
 *                 that row's logp, entropy, loss and gradient NaN.
 *   logp_old    : float[R] behaviour-policy log-probs, or NULL (on-policy).
 *   ref_logp    : float[R] reference-policy log-probs; NULL only if beta == 0.
 *   mask        : uint8[R], nonzero = valid token.
 *   adv         : float[B] or float[R] according to adv_layout.
 *   eps         : clip range, finite, >= 0.   beta, c_ent, grad_scale: finite.
 *   dlogits     : [R, ld] of `dtype`, written (columns >= V untouched), or
 *                 NULL for a forward-only call.  It may be the same pointer as
 *                 logits (in place); any other overlap returns RL_ERR_ALIAS.
 *   logp_out, entropy_out : float[R] written, or NULL.
 *   stats_dev   : one rl_loss_stats in device memory, written at the end.
 *   workspace   : device scratch of workspace_bytes >= rl_policy_loss_workspace_size(R),
 *                 zero-filled before its first use (see above).
 * Deterministic: the same inputs on the same device give bitwise identical
 * outputs (fixed-order fp64 reductions, no floating-point atomics).
 * The launch allows programmatic dependent launch: it may be scheduled while
 * the kernel before it on `stream` is still running, and reads no argument
 * before that kernel has completed.
 */
rl_status rl_policy_loss_fwd_bwd(const void* logits, rl_dtype dtype,
                                 long long B, long long T, long long V, long long ld,
                                 const long long* ids, const float* logp_old,
                                 const float* ref_logp, const unsigned char* mask,
                                 const float* adv, rl_adv_layout adv_layout,
                                 float eps, float beta, float c_ent, float grad_scale,
                                 void* dlogits, float* logp_out, float* entropy_out,
                                 rl_loss_stats* stats_dev,
                                 void* workspace, size_t workspace_bytes, void* stream);

/*
 * Every option of the fused loss, for rl_policy_loss_fwd_bwd_ex.  Fields not
 * listed here mean what they mean for rl_policy_loss_fwd_bwd.  Start from
 * rl_policy_loss_desc_init() so that new fields keep their defaults.
 *
 * Advantages (adv, adv_layout): with RL_ADV_GROUP_REWARDS, adv[B] holds each
 * sequence's reward and the kernel computes, per row, the group-relative
 * advantage A_b = (R_b - mean_g) / (std_g + std_eps) of its group of
 * group_size consecutive sequences (ddof 0 or 1), in fp64 exactly as
 * rl_group_advantages does: reward normalisation and the loss in one launch,
 * as the pages' PPO update kernel fuses advantage estimation into the update
 * (ainews.cool RL.cu article, "PPO 更新内核" bullet).
 *
 * Clip (eps, eps_high): pg = min(r A, clamp(r, 1 - eps, 1 + eps_high) A);
 * eps_high < 0 means eps_high = eps.  A larger eps_high is the asymmetric
 * ("clip-higher") variant.
 *
 * Aggregation (agg, agg_norm): loss = -sum_t w_t J_t and dz scales by
 * grad_scale * w_t, with w_t from rl_loss_agg; L_b = valid tokens of sequence
 * b, B' = sequences with L_b > 0; agg_norm (> 0) is used by
 * RL_AGG_TOKEN_SUM_NORM only.  The statistics pg_term, kl_term, ent_term and
 * clip_frac stay token means (over N) whatever the aggregation.
 */
typedef struct {
  const void* logits;
  rl_dtype dtype;
  long long B, T, V, ld;
  const long long* ids;
  const float* logp_old;         /* nullable */
  const float* ref_logp;         /* nullable iff beta == 0 */
  const unsigned char* mask;
  const float* adv;
  rl_adv_layout adv_layout;
  int group_size;                /* RL_ADV_GROUP_REWARDS: G, B % G == 0, G > ddof */
  int ddof;                      /* RL_ADV_GROUP_REWARDS: 0 or 1 (default 1) */
  double std_eps;                /* RL_ADV_GROUP_REWARDS: default 1e-4 */
  float eps;                     /* default 0.2 */
  float eps_high;                /* default -1 (= eps) */
  float beta, c_ent;             /* default 0 */
  float grad_scale;              /* default 1 */
  rl_loss_agg agg;               /* default RL_AGG_TOKEN_MEAN */
  double agg_norm;               /* RL_AGG_TOKEN_SUM_NORM only */
  void* dlogits;                 /* nullable: forward only */
  float* logp_out;               /* nullable */
  float* entropy_out;            /* nullable */
  rl_loss_stats* stats_dev;
  void* workspace;
  size_t workspace_bytes;
  /* Data parallelism over ranks: device long long[2] = {N, B'} summed over all
   * ranks (see rl_count_tokens), or NULL for this call's own counts.  With it,
   * the gradient scales by the global N (or B'), and loss, pg_term, kl_term,
   * ent_term and clip_frac are this rank's share of the global means (their
   * sum over ranks is the global value); n_tokens stays this rank's count. */
  const long long* global_counts;
  /* Vocabulary parallelism (the LM head split over ranks by vocabulary
   * columns): this call's logits are the columns [vocab_offset,
   * vocab_offset + V) of a vocabulary of vocab_total columns (0 = V), and
   * ids are global.  A row's softmax needs the statistics of every shard, so
   * a step takes two launches per shard with one exchange between them:
   *   1. partials_out != NULL: pass 1 only.  For each valid row, writes
   *      float[4] = (max z, sum 2^((z - max) log2 e), sum 2^(..) (z - max) log2 e,
   *      z_y or -inf when y is not in this shard) at partials_out[4 * row];
   *      nothing else is written (dlogits, logp_out, entropy_out ignored).
   *   2. After gathering the n_shards partial arrays of the shards in order
   *      (shard k at shard_partials[4 * (k * B * T + row)]), shard_partials != NULL:
   *      merges them in shard order, then computes the loss, logp, entropy and
   *      this shard's dlogits columns.  Every shard reports the same loss and
   *      statistics.
   * Both NULL: the ordinary single-shard launch. */
  long long vocab_offset;        /* default 0 */
  long long vocab_total;         /* default 0 (= V) */
  float* partials_out;           /* launch 1: float[4 * B * T], device */
  const float* shard_partials;   /* launch 2: float[4 * n_shards * B * T], device */
  int n_shards;                  /* launch 2: >= 1 */
  /* Launch 2 only (shard_partials != NULL), nullable: each row's gradient
   * coefficients float[4] = (cL, a0, a1, gy) at row_coef_out[4 * row], with
   * which the row's gradient is
   *   dz_v = 2^x (a0 + a1 x) - [v == y] gy,   x = z_v log2(e) - cL,
   * where cL = (max z) log2(e) + log2(sum 2^(..)), a0 = s (g + c_ent H),
   * a1 = s c_ent ln 2 and gy = s g, s being the row's gradient scale
   * (grad_scale w_t); all four are 0 on masked rows.  This is how the
   * tensor-core LM-head backward (rl_lmhead_dlogits) forms the gradient
   * without the logits: the row statistics come from rl_lmhead_row_partials
   * (one shard), and this launch may then have V = 0 columns of its own
   * (logits, ld and dlogits unused; vocab_total > 0 gives the id range). */
  float* row_coef_out;
} rl_policy_loss_desc;

/*
 * Token counts of a batch for data parallelism: counts_dev[0] = N (nonzero
 * mask bytes), counts_dev[1] = B' (sequences of T rows with any valid token).
 * Sum them over ranks (e.g. an all-reduce) and pass them as
 * rl_policy_loss_desc.global_counts so every rank normalises by the global
 * counts; the data path then needs only that 16-byte exchange and, after the
 * loss, a sum of the ranks' loss shares.  mask: uint8[B*T], device;
 * counts_dev: long long[2], device, written.  One launch of one CTA.
 * Errors: RL_ERR_SHAPE (B < 0, T < 0), RL_ERR_NULL.
 */
rl_status rl_count_tokens(const unsigned char* mask, long long B, long long T,
                          long long* counts_dev, void* stream);

/* Fill *desc with the defaults above (all pointers NULL, sizes 0). */
void rl_policy_loss_desc_init(rl_policy_loss_desc* desc);

/*
 * The fused loss with every option of rl_policy_loss_desc, in one launch.
 * rl_policy_loss_fwd_bwd is this call with the defaults (token mean,
 * symmetric clip, advantages given).  Errors as rl_policy_loss_fwd_bwd, plus
 * RL_ERR_NULL for a NULL desc, RL_ERR_DTYPE for an unknown aggregation or
 * layout, RL_ERR_SHAPE for a group size that does not divide B (or is not
 * above ddof), RL_ERR_ARG for ddof not 0/1, a negative/NaN std_eps, a NaN
 * eps_high or a non-positive agg_norm with RL_AGG_TOKEN_SUM_NORM.
 */
rl_status rl_policy_loss_fwd_bwd_ex(const rl_policy_loss_desc* desc, void* stream);

/*
 * rl_policy_loss_fwd_bwd without a caller-provided workspace, for callers
 * that cannot allocate device memory: for example a plug-in inside a host
 * framework that owns the GPU allocator and forbids raw cudaMalloc, or a
 * program that hands all device memory to its own pool at start-up and has
 * no allocation to spare on its update path.  The RL.cu pages have no
 * counterpart to this entry point.
 *
 * Same arguments, meaning and results as rl_policy_loss_fwd_bwd, minus
 * `workspace` and `workspace_bytes`.  The scratch is a file-scope device
 * array of 131,328 bytes inside the library: the status header and one
 * partial per CTA of a persistent grid of up to 2048 CTAs.  The library
 * never plans a larger grid, so the array covers every call; a launch plan
 * that did not fit would return RL_ERR_WORKSPACE.  Every GPU that loads the
 * library holds the array until the process exits.  Nothing is allocated:
 * no cudaMalloc, cudaFree or allocating library call.
 *   - Every call looks up the array's device address (cudaGetSymbolAddress,
 *     with the calling thread's current device and context), so a
 *     cudaDeviceReset or another context on the device is followed
 *     correctly.  The first call on a device also loads the library's device
 *     code there; make that first call before any stream capture.
 *   - Each call clears the array's 256-byte status header with
 *     cudaMemsetAsync on `stream` before launching.  The array keeps the
 *     last call's contents otherwise.
 *   - Every call shares the one array: calls that overlap on the GPU (two
 *     streams, or two host threads) race and give wrong results; serialise
 *     them.  rl_read_device_status does not apply; read device errors from
 *     stats_dev->device_error.
 *   - An argument rejected by rl_policy_loss_fwd_bwd's checks may be reported
 *     after the header was cleared (only the library's own array is written).
 */
rl_status rl_policy_loss_fwd_bwd_noalloc(const void* logits, rl_dtype dtype,
                                         long long B, long long T, long long V, long long ld,
                                         const long long* ids, const float* logp_old,
                                         const float* ref_logp, const unsigned char* mask,
                                         const float* adv, rl_adv_layout adv_layout,
                                         float eps, float beta, float c_ent, float grad_scale,
                                         void* dlogits, float* logp_out, float* entropy_out,
                                         rl_loss_stats* stats_dev, void* stream);

/*
 * Scalar results of rl_value_loss_fwd_bwd (device memory, written at the end).
 *   loss = (1/N) sum_t m_t L_t;  clip_frac = n_clipped / N;
 *   mean_abs_err = (1/N) sum_t m_t |v_t - ret_t|.
 */
typedef struct {
  double loss;
  double clip_frac;
  double mean_abs_err;
  long long n_tokens;
  long long n_clipped;   /* tokens where the clipped square is strictly larger */
} rl_value_stats;

/*
 * PPO clipped value (critic) loss and its gradient with respect to the values.
 * The pages give the PPO loop a critic (ainews.cool RL.cu article, section
 * "技术深度解析", actor/critic bullet); this is the standard clipped form:
 *   vc  = v_old + clamp(v - v_old, -clip_eps, clip_eps)
 *   L_t = 1/2 max((v - ret)^2, (vc - ret)^2)     (1/2 (v - ret)^2 unclipped)
 *   loss = (1/N) sum_t m_t L_t,  N = number of nonzero mask bytes
 *   dvalues_t = grad_scale (m_t / N) * (v - ret)        where the unclipped
 *               square is the larger or equal, else (vc - ret) when
 *               |v - v_old| <= clip_eps, else 0          (inclusive clip)
 *   values, returns : float[n], device, read only (returns from
 *                     rl_gae_reverse_scan);
 *   values_old      : float[n] or NULL; NULL or clip_eps < 0 means unclipped;
 *   mask            : uint8[n], nonzero = valid token;
 *   dvalues         : float[n] written (0 on masked tokens), or NULL;
 *   stats_dev       : one rl_value_stats in device memory.
 * fp32 per token, fp64 fixed-order reduction; one launch of one CTA.
 * Errors: RL_ERR_SHAPE (n < 0), RL_ERR_NULL, RL_ERR_ARG (NaN clip_eps,
 * non-finite grad_scale).  N = 0 gives zeros.
 */
rl_status rl_value_loss_fwd_bwd(const float* values, const float* values_old,
                                const float* returns, const unsigned char* mask, long long n,
                                float clip_eps, float grad_scale, float* dvalues,
                                rl_value_stats* stats_dev, void* stream);

/*
 * Per-row log-softmax statistics of LM-head logits, computed from the hidden
 * states and the LM-head weight without writing the logits.  The actor's
 * logits are its LM-head projection (ainews.cool RL.cu article, section
 * "技术深度解析", actor network with custom matrix multiplication); the
 * behaviour- and reference-policy log-probs the loss takes are these rows'
 * log pi(y_r | .).  For each row r < R, with z_r = hidden_r . W^T (fp32
 * accumulation of the exact products of the 16-bit inputs; the pages' FP16
 * inputs with FP32 accumulation, pitchhut.com RL.cu listing, "Key Features"
 * item 1):
 *   lse_out[r]     = log sum_v exp z_rv
 *   logp_out[r]    = z_r,ids[r] - lse_out[r]     (NaN when ids[r] is outside [0, V))
 *   entropy_out[r] = -sum_v p_rv log p_rv,  p_r = softmax(z_r)
 *   hidden : [R, D] of `dtype` (RL_BF16 or RL_F16), device, row stride ld_h
 *            elements (ld_h >= D), read only;
 *   weight : [V, D] of `dtype`, device, row stride ld_w elements (ld_w >= D),
 *            read only;
 *            both 16-byte aligned, row strides multiples of 8 elements, D a
 *            multiple of 8;
 *   ids    : int64 [R] device;
 *   logp_out, entropy_out, lse_out : float [R] device, each may be NULL;
 *   status_dev : one unsigned int in device memory or NULL; the kernel ORs
 *            RL_DEVERR_ID_RANGE (an id outside [0, V)) or RL_DEVERR_TIMEOUT
 *            (a bounded on-chip wait gave up; outputs are garbage) into it;
 *   workspace : optional device scratch (16-byte aligned) of workspace_bytes,
 *            zero-filled before its first use; every call leaves it
 *            zero-filled again, except one that timed out.  With it the
 *            launch may cut the vocabulary into slices so that the work
 *            spreads evenly over the SMs (see rl_lmhead_workspace_size); NULL
 *            or too small a workspace gives the unsliced launch, with the same
 *            results up to fp32 rounding order.  Calls sharing a workspace
 *            must not overlap on the GPU.
 * One launch of a persistent tensor-core kernel (tcgen05, TMA, tensor memory).
 * Allocates nothing; stream-ordered.  Errors: RL_ERR_DTYPE (not RL_BF16 or
 * RL_F16), RL_ERR_SHAPE (R < 0, R >= 2^31,
 * V < 1, V > 2^31, D < 8, D not a multiple of 8, a stride below D),
 * RL_ERR_NULL, RL_ERR_ALIGN, RL_ERR_CUDA.  R == 0 launches nothing.
 */
rl_status rl_lmhead_logprobs(const void* hidden, long long ld_h, const void* weight, long long ld_w,
                             rl_dtype dtype, long long R, long long D, long long V,
                             const long long* ids,
                             float* logp_out, float* entropy_out, float* lse_out,
                             unsigned int* status_dev, void* workspace, size_t workspace_bytes,
                             void* stream);

/*
 * rl_lmhead_logprobs with each row's partial softmax statistics as output,
 * in the form the loss's merge launch takes (rl_policy_loss_desc
 * .shard_partials with n_shards = 1): float[4] at partials_out[4 * r] =
 *   (m, s, t, z_y) with m = max_v z_rv, s = sum_v 2^x, t = sum_v 2^x x,
 *   x = (z_rv - m) log2(e), and z_y the sampled id's logit (-inf when ids[r]
 *   is outside [0, V)),
 * so lse = m + ln s and H = ln 2 (log2 s - t / s).  Same kernel, arguments,
 * workspace, status bits and errors as rl_lmhead_logprobs; partials_out is
 * device float[4 * R], 16-byte aligned (RL_ERR_NULL / RL_ERR_ALIGN).  This is
 * the first step of the policy loss through the LM head without the logits:
 * then the merge launch with row_coef_out, then rl_lmhead_dlogits,
 * rl_lmhead_dhidden and rl_lmhead_dweight.
 */
rl_status rl_lmhead_row_partials(const void* hidden, long long ld_h, const void* weight,
                                 long long ld_w, rl_dtype dtype, long long R, long long D,
                                 long long V, const long long* ids, float* partials_out,
                                 unsigned int* status_dev, void* workspace,
                                 size_t workspace_bytes, void* stream);

/*
 * The loss gradient with respect to the LM-head logits, formed from the
 * hidden states on the tensor cores without the logits ever being written:
 * the logits tile z = hidden . W^T (fp32 accumulation of the 16-bit
 * products, as for rl_lmhead_logprobs) is recomputed in tensor memory and
 * the epilogue writes, for each row r < R and column v < V,
 *   dlogits[r, v] = 2^x (a0 + a1 x) - [v == ids[r]] gy,   x = z_rv log2(e) - cL
 * rounded to `dtype`, with (cL, a0, a1, gy) = row_coef[4 * r .. 4 * r + 3] the
 * row's coefficients from the loss's merge launch (rl_policy_loss_desc
 * .row_coef_out).  That is the fused loss's gradient
 *   s [ g (p_v - [v = y]) + c_ent p_v (log p_v + H) ]
 * (the pages' PPO update kernel: ainews.cool RL.cu article, section
 * "技术深度解析", bullet "PPO 更新内核"; the actor's own matrix multiplication:
 * the same section's policy and value networks bullet).  A row whose a0 and
 * a1 are both 0 (masked rows) gets only the -gy term (0 for masked rows).
 *   hidden, weight, ids : as rl_lmhead_logprobs;
 *   row_coef : float[4 * R] device, 16-byte aligned, read only;
 *   dlogits  : [R, ld_dz] of `dtype`, device, 16-byte aligned, ld_dz >= V a
 *              multiple of 8 elements; columns V .. ld_dz-1 are not written;
 *   status_dev : as rl_lmhead_logprobs (RL_DEVERR_TIMEOUT).
 * One launch of a persistent tensor-core kernel (tcgen05, TMA, tensor
 * memory); allocates nothing; stream-ordered.  Errors: RL_ERR_DTYPE,
 * RL_ERR_SHAPE (R < 0, R >= 2^31, V < 1, V >= 2^31, D < 8 or not a multiple
 * of 8, a stride below its row or not a multiple of 8 elements), RL_ERR_NULL,
 * RL_ERR_ALIGN, RL_ERR_CUDA.  R == 0 launches nothing.
 */
rl_status rl_lmhead_dlogits(const void* hidden, long long ld_h, const void* weight, long long ld_w,
                            rl_dtype dtype, long long R, long long D, long long V,
                            const long long* ids, const float* row_coef, void* dlogits,
                            long long ld_dz, unsigned int* status_dev, void* stream);

/*
 * Gradient with respect to the hidden states through the LM head:
 *   dhidden[r, d] = sum_v dlogits[r, v] weight[v, d]
 * (the backward of the actor's LM-head matrix multiplication, ainews.cool
 * RL.cu article, section "技术深度解析", policy and value networks bullet),
 * on the tensor cores with fp32 accumulation of the exact 16-bit products,
 * rounded once to `dtype`.
 *   dlogits : [R, ld_dz] of `dtype`, device, read only (ld_dz >= V);
 *   weight  : [V, ld_w] of `dtype`, device, read only (ld_w >= D);
 *   dhidden : [R, ld_dh] of `dtype`, device, written (ld_dh >= D);
 *   strides multiples of 8 elements, bases 16-byte aligned; status_dev as
 *   rl_lmhead_logprobs.  Errors as rl_lmhead_dlogits.  R == 0 launches nothing.
 */
rl_status rl_lmhead_dhidden(const void* dlogits, long long ld_dz, const void* weight, long long ld_w,
                            rl_dtype dtype, long long R, long long D, long long V, void* dhidden,
                            long long ld_dh, unsigned int* status_dev, void* stream);

/*
 * Gradient with respect to the LM-head weight:
 *   dweight[v, d] (+)= sum_r dlogits[r, v] hidden[r, d]
 * (the same backward, for the weight), on the tensor cores with fp32
 * accumulation of the exact 16-bit products; fp32 output.  accumulate != 0
 * adds the product to what dweight holds (a batch taken in chunks of rows),
 * 0 overwrites it.
 *   dlogits : [R, ld_dz] of `dtype`, device, read only;
 *   hidden  : [R, ld_h] of `dtype`, device, read only;
 *   dweight : float [V, ld_dw], device, 16-byte aligned, ld_dw >= D a
 *             multiple of 4;
 *   status_dev as rl_lmhead_logprobs.  Errors as rl_lmhead_dlogits.  R == 0
 *   leaves dweight as it is (accumulate) or zero (overwrite).
 */
rl_status rl_lmhead_dweight(const void* dlogits, long long ld_dz, const void* hidden, long long ld_h,
                            rl_dtype dtype, long long R, long long D, long long V, float* dweight,
                            long long ld_dw, int accumulate, unsigned int* status_dev, void* stream);

/*
 * Workspace bytes rl_lmhead_logprobs needs for its best work split of R rows
 * over V on the current device (0 when the unsliced launch is already the
 * best, or the shape is invalid, or no device answers).  Host-only query.
 */
size_t rl_lmhead_workspace_size(long long R, long long V);

/*
 * The work split rl_lmhead_logprobs would use with workspace_bytes of
 * workspace on a GPU of sm_count SMs (sm_count < 1: the current device):
 * vocabulary slices per 128-row tile, CTAs in the persistent grid, row
 * tiles per unit group (units run slice by slice inside a group, so the
 * hidden tiles in use at one time stay in L2) and the workspace bytes that
 * split uses (0 when unsliced).  Any output pointer may be NULL.  Host-only;
 * with sm_count >= 1 it needs no GPU.  Errors: RL_ERR_SHAPE (R < 1 or as
 * rl_lmhead_logprobs), RL_ERR_CUDA.
 */
rl_status rl_lmhead_plan(long long R, long long D, long long V, size_t workspace_bytes, int sm_count,
                         int* n_slices, int* grid, int* group, size_t* workspace_needed);

/*
 * The launch shape rl_policy_loss_fwd_bwd would use on the current device for
 * this row shape: CTAs per cluster (always 1: each CTA holds whole rows),
 * CTAs in the persistent grid and dynamic shared memory per CTA.  Rows of
 * more than 100 KB (V * element size) run one 608-thread CTA per SM; shorter
 * rows run two 320-thread CTAs per SM, so n_clusters is twice the SM count
 * there.
 * Host-only query.  Errors as for rl_policy_loss_fwd_bwd's shape checks.
 */
rl_status rl_policy_loss_launch_shape(rl_dtype dtype, long long V, long long n_rows,
                                      int* cluster_size, int* n_clusters, int* smem_bytes);

/*
 * Synchronises `stream`, then reads the device status word the last
 * rl_policy_loss_fwd_bwd call on `workspace` left: RL_OK, RL_ERR_ID_RANGE or
 * RL_ERR_TIMEOUT (the first of the bits set), or RL_ERR_CUDA.
 */
rl_status rl_read_device_status(const void* workspace, void* stream);

/*
 * Self-test of failure detection, without a fault: every wait on an on-chip
 * barrier in this library's kernels is bounded, and a wait that runs out
 * raises RL_DEVERR_TIMEOUT and lets the kernel return normally, so the CUDA
 * context stays usable.  This call runs that same bounded wait, for
 * limit_ns nanoseconds, on a barrier that nothing completes: one thread of
 * one CTA waits, gives up, ORs RL_DEVERR_TIMEOUT into *status_dev (one
 * unsigned int in device memory) and writes the nanoseconds it waited to
 * *waited_ns_dev (device, may be NULL).  The pages have no counterpart; it
 * exists so that tests can check the timeout path on a GPU.
 * Errors: RL_ERR_NULL (status_dev), RL_ERR_ARG (limit_ns outside
 * [1 us, 10 s]), RL_ERR_CUDA.
 */
rl_status rl_selftest_wait_timeout(unsigned long long limit_ns, unsigned int* status_dev,
                                   unsigned long long* waited_ns_dev, void* stream);

/* A static, human-readable name for a status code. */
const char* rl_status_string(rl_status status);

#ifdef __cplusplus
}
#endif

#endif /* RLLOSS_H */
