"""Plain fp64 CPU oracle for the fused RL policy-loss step.

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg may import this package.  The CUDA library never
loads it and shares no code with it: the heavy per-row loops live in
``rlref.c`` (built here with gcc, no fast-math, no FMA contraction) and the
per-token objective is numpy in float64.

Sources.  The three pages on RL.cu ("LLM Reinforcement Learning in Pure CUDA")
name the parts of the update without writing their formulas:

* pitchhut.com RL.cu listing, "Project Highlights" and "Key Features" item 3:
  the method is GRPO (group relative policy optimisation) alongside SFT;
* mlllm.io RL.cu article, section "Что произошло": the full SFT + GRPO loop;
* ainews.cool RL.cu article, section "技术深度解析" (technical deep dive):
  the rollout buffer holds states, actions, rewards and log-probabilities;
  the "PPO 更新内核" (PPO update kernel) bullet fuses advantage estimation,
  the clipped surrogate objective and the entropy bonus into one launch; the
  paragraph after the benchmark table adds a KL penalty against policy
  collapse and reward normalisation.

Each function below states the standard definition it writes out for the part
the pages name.  Readings taken where the pages are silent:

* group advantage: A = (R - mean_g) / (std_g + 1e-4) with the unbiased
  (ddof = 1) standard deviation; ddof = 0 is a flag;
* GAE: terminal bootstrap value 0 at the end of each sequence, no whitening;
* KL: the k3 estimator exp(d) - d - 1 with d = ref_logp - logp;
* masked mean: one global token mean, loss = -(1/N) sum_t m_t J_t, N = sum m;
  N = 0 gives loss 0 and an all-zero gradient;
* clip gradient: flows at r = 1 +/- eps exactly (inclusive boundary);
* no ``logp_old`` means on-policy (r = 1, dr/dlogp = 1); no ``ref_logp`` means
  no KL term.
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "rlref.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_SO = os.path.join(_OUT_DIR, "librlref.so")

F32, BF16, F16, F64 = 0, 1, 2, 3
DTYPE_CODES = {"f32": F32, "bf16": BF16, "f16": F16, "f64": F64}
STORAGE = {F32: np.float32, BF16: np.uint16, F16: np.uint16, F64: np.float64}

_lib_handle = None


def build(force: bool = False) -> str:
    """Compile rlref.c into a shared object next to it (plain C11, -O2)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math",
                               "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _SO)
    return _SO


def _lib():
    global _lib_handle
    if _lib_handle is None:
        lib = ctypes.CDLL(build())
        P, LL, I, D = ctypes.c_void_p, ctypes.c_longlong, ctypes.c_int, ctypes.c_double
        lib.rlref_decode.argtypes = [P, I, LL, P]
        lib.rlref_encode.argtypes = [P, LL, I, P]
        lib.rlref_count.argtypes = [P, LL]
        lib.rlref_count.restype = LL
        lib.rlref_row_stats.argtypes = [P, I, LL, LL, P, P, LL, LL, P, P, P]
        lib.rlref_dlogits_rows.argtypes = [P, I, LL, LL, P, P, LL, P, P, P, P, D, I, P, LL]
        _lib_handle = lib
    return _lib_handle


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def _code(dtype) -> int:
    return DTYPE_CODES[dtype] if isinstance(dtype, str) else int(dtype)


def default_threads() -> int:
    return len(os.sched_getaffinity(0))


# --------------------------------------------------------------------------- formats
def decode(storage: np.ndarray, dtype) -> np.ndarray:
    """Exact decode of bf16/f16 (uint16 storage), f32 or f64 elements to float64."""
    src = np.ascontiguousarray(storage)
    out = np.empty(src.shape, np.float64)
    _lib().rlref_decode(_ptr(src), _code(dtype), src.size, _ptr(out))
    return out


def encode(x: np.ndarray, dtype) -> np.ndarray:
    """Round float64 values once to ``dtype`` (round to nearest even, subnormals kept)."""
    code = _code(dtype)
    src = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty(src.shape, STORAGE[code])
    _lib().rlref_encode(_ptr(src), src.size, code, _ptr(out))
    return out


def ulp(x: np.ndarray, dtype) -> np.ndarray:
    """Spacing of ``dtype`` at |x| (the subnormal quantum below the normal range)."""
    p, emin = {F32: (24, -126), BF16: (8, -126), F16: (11, -14), F64: (53, -1022)}[_code(dtype)]
    a = np.abs(np.asarray(x, np.float64))
    _, k = np.frexp(a)
    lead = np.maximum(k - 1, emin)
    return np.ldexp(1.0, lead - (p - 1))


# --------------------------------------------------------------------------- advantages
def group_advantages(rewards: np.ndarray, group_size: int, std_eps: float = 1e-4,
                     ddof: int = 1) -> np.ndarray:
    """Group-relative advantage (GRPO reward normalisation).

    Pages: pitchhut.com RL.cu listing, "Key Features" item 3 (GRPO) and the
    ainews.cool article's "reward normalisation" sentence after its benchmark
    table.  Sequences are group-major: sequence i = g * G + j.  For each
    group, mean and standard deviation (ddof 1 by default) of its G rewards,
    then A_i = (R_i - mean) / (std + std_eps).
    """
    R = np.asarray(rewards, np.float64).reshape(-1)
    G = int(group_size)
    if G <= 0 or R.size % G:
        raise ValueError("rewards length must be a multiple of group_size")
    if G - ddof <= 0:
        raise ValueError("group_size must exceed ddof")
    A = np.empty_like(R)
    for g in range(R.size // G):
        grp = R[g * G:(g + 1) * G]
        mean = sum(grp) / G
        var = sum((x - mean) ** 2 for x in grp) / (G - ddof)
        std = math.sqrt(var)
        A[g * G:(g + 1) * G] = [(x - mean) / (std + std_eps) for x in grp]
    return A


def gae(rewards: np.ndarray, values: np.ndarray, lengths: np.ndarray,
        gamma: float, lam: float):
    """Generalised advantage estimation by a reverse scan over time.

    Page: ainews.cool RL.cu article, "PPO 更新内核" bullet (advantage
    estimation inside the PPO update) and the actor/critic bullet before it.
    For a sequence of length L, walking t = L-1 down to 0:
        delta_t = r_t + gamma * V_{t+1} - V_t      (V_L = 0: the episode ends)
        A_t     = delta_t + gamma * lam * A_{t+1}  (A_L = 0)
        ret_t   = A_t + V_t
    Positions t >= L get A = ret = 0; lengths are clamped to [0, T].
    """
    r = np.asarray(rewards, np.float64)
    v = np.asarray(values, np.float64)
    B, T = r.shape
    A = np.zeros((B, T))
    ret = np.zeros((B, T))
    for b in range(B):
        L = min(max(int(lengths[b]), 0), T)
        nxt_v, nxt_a = 0.0, 0.0
        for t in range(L - 1, -1, -1):
            delta = r[b, t] + gamma * nxt_v - v[b, t]
            a = delta + gamma * lam * nxt_a
            A[b, t] = a
            ret[b, t] = a + v[b, t]
            nxt_v, nxt_a = v[b, t], a
    return A, ret


# --------------------------------------------------------------------------- loss
def count(mask: np.ndarray) -> int:
    """N = number of valid tokens (nonzero mask bytes)."""
    m = np.ascontiguousarray(mask, dtype=np.uint8)
    return int(_lib().rlref_count(_ptr(m), m.size))


def row_stats(logits: np.ndarray, dtype, V: int, ids: np.ndarray, mask: np.ndarray,
              threads: int | None = None):
    """Per-row lse, logp of the sampled id and entropy (log-softmax over V).

    ``logits`` is a 2-D array [rows, ld] of the element storage (uint16 for
    bf16/f16).  Rows with mask 0 give zeros.  Rows are split over threads; the
    arithmetic of each row is the sequential loop in rlref.c.
    """
    lg = np.ascontiguousarray(logits)
    n_rows, ld = lg.shape
    ids = np.ascontiguousarray(ids, dtype=np.int64)
    m = np.ascontiguousarray(mask, dtype=np.uint8)
    lse, logp, ent = (np.zeros(n_rows) for _ in range(3))
    lib, code = _lib(), _code(dtype)
    threads = threads or default_threads()
    step = max(1, -(-n_rows // (threads * 4)))

    def work(r0):
        lib.rlref_row_stats(_ptr(lg), code, ld, V, _ptr(ids), _ptr(m), r0, min(n_rows, r0 + step),
                            _ptr(lse), _ptr(logp), _ptr(ent))

    if threads == 1 or n_rows <= step:
        for r0 in range(0, n_rows, step):
            work(r0)
    else:
        with ThreadPoolExecutor(threads) as ex:
            list(ex.map(work, range(0, n_rows, step)))
    return lse, logp, ent


def surrogate(r, A, eps, eps_high=None):
    """Clipped surrogate pg = min(r A, clip(r, 1 - eps, 1 + eps_high) A) and its
    derivative with respect to logp (r = exp(logp - logp_old), dr/dlogp = r).

    Page: ainews.cool RL.cu article, "PPO 更新内核" bullet (clipped surrogate
    objective).  eps_high (default eps) is the upper clip offset; a larger
    upper than lower offset is the asymmetric ("clip-higher") variant.  Where
    the two branches differ, the smaller is the clipped one exactly when
    (A > 0 and r > 1 + eps_high) or (A < 0 and r < 1 - eps); its derivative
    is 0 there and r A elsewhere (ties, including r on a boundary, take r A).
    Returns (pg, dpg, clipped).
    """
    hi = 1.0 + (eps if eps_high is None else eps_high)
    lo = 1.0 - eps
    r = np.asarray(r, np.float64)
    A = np.asarray(A, np.float64)
    s1 = r * A
    s2 = np.clip(r, lo, hi) * A
    pg = np.minimum(s1, s2)
    clipped = ((A > 0) & (r > hi)) | ((A < 0) & (r < lo))
    dpg = np.where(clipped, 0.0, r * A)
    return pg, dpg, clipped


def token_objective(logp, ent, mask, adv, logp_old, ref_logp, eps, beta, c_ent, eps_high=None):
    """Per-token PPO/GRPO objective J_t and its derivative g_t = dJ_t/dlogp_t.

    Page: ainews.cool RL.cu article, "PPO 更新内核" bullet (clipped surrogate,
    entropy bonus) and the KL-penalty sentence after the benchmark table.
        r   = exp(logp - logp_old)                (r = 1 without logp_old)
        pg  = min(r A, clip(r, 1 - eps, 1 + eps) A)
        kl  = exp(d) - d - 1,  d = ref - logp     (k3 estimator; 0 without ref)
        J   = pg - beta kl + c_ent H
    Derivative with respect to logp: pg' = r A, except 0 when the clipped
    branch is strictly the smaller one, i.e. (A > 0 and r > 1 + eps) or
    (A < 0 and r < 1 - eps); kl' = 1 - exp(d); so g = pg' + beta (exp(d) - 1).
    Masked tokens give zeros everywhere.

    Also returned: both one-sided derivatives of the surrogate at every token,
    g_unclipped (pg' = r A) and g_clipped (pg' = 0), each with the same KL
    term.  At a token whose ratio lies on a clip boundary the surrogate has a
    kink; there each of the two is a valid gradient, and an implementation
    that evaluates r in lower precision may take either side.
    """
    m = np.asarray(mask).astype(bool)
    logp = np.where(m, logp, 0.0)
    A = np.where(m, np.asarray(adv, np.float64), 0.0)
    r = np.exp(logp - np.where(m, logp_old, 0.0)) if logp_old is not None else np.ones_like(logp)
    r = np.where(m, r, 1.0)
    pg, dpg, clipped = surrogate(r, A, eps, eps_high)
    if ref_logp is not None:
        d = np.where(m, np.asarray(ref_logp, np.float64) - logp, 0.0)
        kl = np.exp(d) - d - 1.0
        dkl = np.exp(d) - 1.0
    else:
        kl = np.zeros_like(logp)
        dkl = np.zeros_like(logp)
    H = np.where(m, ent, 0.0)
    J = pg - beta * kl + c_ent * H
    g = dpg + beta * dkl
    z = lambda x: np.where(m, x, 0.0)
    return dict(r=z(r), pg=z(pg), kl=z(kl), H=H, J=z(J), g=z(g), clipped=m & clipped,
                g_unclipped=z(r * A + beta * dkl), g_clipped=z(beta * dkl))


AGGREGATIONS = ("token_mean", "seq_mean_token_mean", "seq_mean_token_sum", "token_sum_norm")


def loss_weights(mask, T, agg="token_mean", agg_norm=None, global_counts=None):
    """Weight w_t of each token in loss = -sum_t w_t J_t (0 on masked tokens).

    The pages name the masked loss only as the PPO/GRPO objective; the four
    aggregations in use for it are:
      token_mean          w = 1 / N                  (one mean over all tokens)
      seq_mean_token_mean w = 1 / (B' L_b)           (mean over sequences of
                                                      each sequence's token mean)
      seq_mean_token_sum  w = 1 / B'                 (mean over sequences of
                                                      each sequence's token sum)
      token_sum_norm      w = 1 / agg_norm           (token sum over a fixed
                                                      normaliser, e.g. B * T_max)
    L_b = valid tokens of sequence b (row b*T + t); B' = sequences with L_b > 0.
    With ``global_counts`` = (N, B') of a whole data-parallel batch, of which
    ``mask`` is one rank's share, N and B' are those totals.
    """
    m = np.asarray(mask, dtype=np.uint8).reshape(-1) != 0
    w = np.zeros(m.size)
    if agg == "token_mean":
        N = int(m.sum()) if global_counts is None else int(global_counts[0])
        w[m] = 1.0 / N if N else 0.0
    elif agg in ("seq_mean_token_mean", "seq_mean_token_sum"):
        L = m.reshape(-1, T).sum(axis=1)
        Bp = int((L > 0).sum()) if global_counts is None else int(global_counts[1])
        Lrow = np.repeat(L, T)
        if agg == "seq_mean_token_mean":
            w[m] = 1.0 / (Bp * Lrow[m])
        else:
            w[m] = 1.0 / Bp
    elif agg == "token_sum_norm":
        w[m] = 1.0 / float(agg_norm)
    else:
        raise ValueError(agg)
    return w


def loss_from_stats(logp, ent, mask, adv_row, logp_old=None, ref_logp=None, eps=0.2,
                    beta=0.0, c_ent=0.0, eps_high=None, agg="token_mean", T=None,
                    agg_norm=None, global_counts=None):
    """Loss and monitoring statistics from per-row (logp, H) (fp64, math.fsum sums).

    loss = -sum_t w_t J_t with the weights of ``loss_weights`` (token_mean:
    -(1/N) sum_t m_t J_t); pg_term, kl_term, ent_term are the token means of
    pg, kl and H whatever the aggregation; n_clipped the tokens whose
    surrogate gradient the clip cuts.  N = 0 gives zeros.  Also returns the
    per-token arrays of token_objective and the weights.
    """
    m = np.ascontiguousarray(mask, dtype=np.uint8).reshape(-1)
    N = count(m)                      # this call's valid tokens
    Nd = N if global_counts is None else int(global_counts[0])  # the means' denominator
    obj = token_objective(logp, ent, m, adv_row, logp_old, ref_logp, eps, beta, c_ent, eps_high)
    mb = m.astype(bool)
    T = m.size if T is None else T
    w = loss_weights(m, T, agg, agg_norm, global_counts) if N else np.zeros(m.size)
    if N > 0:
        if agg == "token_mean":
            loss = -math.fsum(obj["J"][mb]) / Nd
        else:
            loss = -math.fsum((w * obj["J"])[mb])
        pg_term = math.fsum(obj["pg"][mb]) / Nd
        kl_term = math.fsum(obj["kl"][mb]) / Nd
        ent_term = math.fsum(obj["H"][mb]) / Nd
    else:
        loss = pg_term = kl_term = ent_term = 0.0
    n_clipped = int(obj["clipped"].sum())
    return dict(loss=loss, pg_term=pg_term, kl_term=kl_term, ent_term=ent_term, n_tokens=N,
                n_clipped=n_clipped, clip_frac=(n_clipped / Nd if N else 0.0),
                logp=np.where(mb, logp, 0.0), entropy=np.where(mb, ent, 0.0), weights=w, **obj)


def policy_loss(logits, dtype, V, ids, mask, adv_row, logp_old=None, ref_logp=None,
                eps=0.2, beta=0.0, c_ent=0.0, grad_scale=1.0, grad_rows=None,
                out_dtype=None, threads=None, eps_high=None, agg="token_mean", T=None,
                agg_norm=None):
    """The whole fused step on CPU: loss, statistics, per-row outputs and dlogits.

    ``adv_row`` is the advantage of each row (a per-sequence advantage already
    broadcast over its T positions).  ``grad_rows`` lists the rows whose
    logits gradient is wanted (all rows if None, none if False); the gradient
    is returned in ``out_dtype`` (default: the logits' format) as rows
    [len(grad_rows), V].

    Loss = -sum_t w_t J_t (token_mean: w_t = m_t / N); N = 0 gives loss 0 and
    zero gradients.
    dz_v = grad_scale w_t [ g_t (p_v - [v = y_t]) + c_ent p_v (ln p_v + H_t) ]
    (d logp / dz_v = [v = y] - p_v and dH / dz_v = -p_v (ln p_v + H)).
    """
    lg = np.ascontiguousarray(logits)
    n_rows = lg.shape[0]
    m = np.ascontiguousarray(mask, dtype=np.uint8).reshape(-1)
    ids = np.ascontiguousarray(ids, dtype=np.int64).reshape(-1)
    lse, logp, ent = row_stats(lg, dtype, V, ids, m, threads)
    out = loss_from_stats(logp, ent, m, adv_row, logp_old, ref_logp, eps, beta, c_ent,
                          eps_high, agg, T, agg_norm)
    out["lse"] = lse
    if grad_rows is not False:
        rows = np.arange(n_rows, dtype=np.int64) if grad_rows is None else \
            np.ascontiguousarray(grad_rows, dtype=np.int64)
        scale = np.where(m[rows] != 0, grad_scale * out["weights"][rows], 0.0)
        out["grad_rows"] = rows
        out["dlogits"] = dlogits_rows(lg, dtype, V, ids, rows, lse[rows], ent[rows],
                                      out["g"][rows], scale, c_ent,
                                      out_dtype if out_dtype is not None else dtype, threads)
    return out


def dlogits_rows(logits, dtype, V, ids, rows, lse, ent, g, scale, c_ent, out_dtype,
                 threads=None):
    """dz for the listed rows; see rlref.c for the formula (one row per call site)."""
    lg = np.ascontiguousarray(logits)
    ld = lg.shape[1]
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    arrs = [np.ascontiguousarray(a, dtype=np.float64) for a in (lse, ent, g, scale)]
    ocode = _code(out_dtype)
    out = np.zeros((rows.size, V), STORAGE[ocode])
    ids = np.ascontiguousarray(ids, dtype=np.int64)
    lib, code = _lib(), _code(dtype)
    threads = threads or default_threads()
    step = max(1, -(-rows.size // (threads * 4)))

    def work(i0):
        i1 = min(rows.size, i0 + step)
        sub = [np.ascontiguousarray(a[i0:i1]) for a in arrs]
        r = np.ascontiguousarray(rows[i0:i1])
        o = out[i0:i1]
        lib.rlref_dlogits_rows(_ptr(lg), code, ld, V, _ptr(ids), _ptr(r), r.size,
                               _ptr(sub[0]), _ptr(sub[1]), _ptr(sub[2]), _ptr(sub[3]),
                               float(c_ent), ocode, o.ctypes.data, V)

    if threads == 1 or rows.size <= step:
        for i0 in range(0, rows.size, step):
            work(i0)
    else:
        with ThreadPoolExecutor(threads) as ex:
            list(ex.map(work, range(0, rows.size, step)))
    return out


# --------------------------------------------------------------------------- critic
def value_loss(values, values_old, returns, mask, clip_eps=None, grad_scale=1.0):
    """PPO clipped value (critic) loss and its gradient with respect to the values.

    Page: ainews.cool RL.cu article, section "技术深度解析": the policy (actor)
    and value (critic) networks of the PPO loop; the value loss itself is not
    written there, so this is the standard clipped form:
        vc  = v_old + clip(v - v_old, -clip_eps, clip_eps)
        L_t = 1/2 max((v - ret)^2, (vc - ret)^2)          (unclipped if no v_old
                                                           or clip_eps is None)
        loss = (1/N) sum_t m_t L_t
    dL/dv_t = grad_scale (m_t / N) * ((v - ret) where the unclipped square is
    the larger or equal, else (vc - ret) [|v - v_old| <= clip_eps]); the clip
    is inclusive at the boundary.  N = 0 gives zeros.
    Returns dict(loss, dvalues, n_tokens, n_clipped, clip_frac, mean_abs_err);
    n_clipped counts tokens where the clipped square is strictly larger.
    """
    v = np.asarray(values, np.float64).reshape(-1)
    ret = np.asarray(returns, np.float64).reshape(-1)
    m = np.asarray(mask).reshape(-1) != 0
    N = int(m.sum())
    u = (v - ret) ** 2
    if values_old is not None and clip_eps is not None:
        vo = np.asarray(values_old, np.float64).reshape(-1)
        vc = vo + np.clip(v - vo, -clip_eps, clip_eps)
        c = (vc - ret) ** 2
        inside = np.abs(v - vo) <= clip_eps
        use_c = c > u
        grad = np.where(use_c, (vc - ret) * inside, v - ret)
        L = 0.5 * np.maximum(u, c)
    else:
        use_c = np.zeros(v.size, bool)
        grad = v - ret
        L = 0.5 * u
    if N == 0:
        return dict(loss=0.0, dvalues=np.zeros(v.size), n_tokens=0, n_clipped=0, clip_frac=0.0,
                    mean_abs_err=0.0)
    loss = math.fsum(L[m]) / N
    dvalues = np.where(m, grad_scale * grad / N, 0.0)
    n_clipped = int((use_c & m).sum())
    return dict(loss=loss, dvalues=dvalues, n_tokens=N, n_clipped=n_clipped,
                clip_frac=n_clipped / N, mean_abs_err=math.fsum(np.abs(v - ret)[m]) / N)


def masked_whiten(x, mask, eps=1e-8, shift_mean=True):
    """Masked advantage whitening over the valid tokens of a batch.

    The pages name advantage estimation and reward normalisation as parts of
    the update (ainews.cool RL.cu article, "PPO 更新内核" bullet and the
    paragraph after the benchmark table); the usual normalisation of PPO-GAE
    advantages is this one:
        mu  = (1/N) sum_t m_t x_t,  var = (1/(N-1)) sum_t m_t (x_t - mu)^2
        out = (x - mu) / sqrt(var + eps)      (x / sqrt(var + eps) without the
                                               mean shift), 0 on masked tokens
    N < 2 gives x - mu (or x) divided by sqrt(eps): var is taken as 0.
    """
    x = np.asarray(x, np.float64).reshape(-1)
    m = np.asarray(mask).reshape(-1) != 0
    N = int(m.sum())
    if N == 0:
        return np.zeros(x.size)
    mu = math.fsum(x[m]) / N
    var = math.fsum((x[m] - mu) ** 2) / (N - 1) if N > 1 else 0.0
    out = ((x - mu) if shift_mean else x) / math.sqrt(var + eps)
    return np.where(m, out, 0.0)


# --------------------------------------------------------------------------- LM head
def lmhead_row_stats(hidden, weight, ids, dtype="bf16", threads=None):
    """Log-softmax statistics of logits = hidden @ weight^T, never rounded.

    The logits the fused policy loss consumes come from the policy's LM head
    (ainews.cool RL.cu article, "技术深度解析": the actor network with its
    custom matrix multiplication); this is that projection followed by the row
    statistics of ``row_stats``: a library matmul in float64 on the exactly
    decoded bf16/fp16 inputs, then lse, logp of the sampled id and entropy.
    hidden: [R, D], weight: [V, D] (element storage); returns (lse, logp, H).
    """
    Hm = decode(np.ascontiguousarray(hidden), dtype)
    Wm = decode(np.ascontiguousarray(weight), dtype)
    logits = Hm @ Wm.T
    ids = np.ascontiguousarray(ids, dtype=np.int64).reshape(-1)
    return row_stats(logits, F64, Wm.shape[0], ids, np.ones(logits.shape[0], np.uint8), threads)


def lmhead_logits(hidden, weight, dtype="bf16"):
    """Logits = hidden @ weight^T in float64 on the exactly decoded 16-bit
    inputs (a library matmul), never rounded.  hidden [R, D], weight [V, D]."""
    Hm = decode(np.ascontiguousarray(hidden), dtype)
    Wm = decode(np.ascontiguousarray(weight), dtype)
    return Hm @ Wm.T


def lmhead_policy_loss(hidden, weight, dtype, ids, mask, adv_row, logp_old=None, ref_logp=None,
                       eps=0.2, beta=0.0, c_ent=0.0, grad_scale=1.0, eps_high=None,
                       agg="token_mean", T=None, agg_norm=None, threads=None):
    """The policy loss from hidden states and its gradients, all in float64.

    The actor's logits are its LM-head projection (ainews.cool RL.cu article,
    "技术深度解析", policy and value networks bullet), so by the chain rule
      z  = hidden @ W^T                         (lmhead_logits)
      dz = dL/dz  of policy_loss on z           (row_stats, loss_from_stats,
                                                 dlogits_rows with no rounding)
      dhidden = dz @ W,   dW = dz^T @ hidden    (library matmuls)
    with every step the plain definition and nothing rounded.  Returns the
    policy_loss outputs plus z, dz (float64 [R, V]), dhidden and dweight.
    """
    z = lmhead_logits(hidden, weight, dtype)
    R, V = z.shape
    m = np.ascontiguousarray(mask, dtype=np.uint8).reshape(-1)
    ids = np.ascontiguousarray(ids, dtype=np.int64).reshape(-1)
    out = policy_loss(z, F64, V, ids, m, adv_row, logp_old, ref_logp, eps, beta, c_ent,
                      grad_scale, None, F64, threads, eps_high, agg, T, agg_norm)
    dz = out["dlogits"]
    Hm = decode(np.ascontiguousarray(hidden), dtype)
    Wm = decode(np.ascontiguousarray(weight), dtype)
    out.update(z=z, dz=dz, dhidden=dz @ Wm, dweight=dz.T @ Hm)
    return out
