"""Python binding of librlloss, the GB300-native fused RL policy-loss library.

Argument marshalling only: every function forwards to the C entry point of
the same name declared in include/rlloss.h, with the same arguments in the
same order.  Array arguments may be torch CUDA tensors (their data_ptr() is
passed), plain integer device addresses, or None for NULL.  ``stream`` may be
a torch.cuda.Stream, an integer cudaStream_t, or None for torch's current
stream.  A status other than RL_OK raises RlLossError.

There is no fallback: if librlloss.so has not been built (``build()``), every
call raises.
"""
from __future__ import annotations

import ctypes
import os

from ._build import LIB_PATH, build

RL_OK, RL_ERR_NULL, RL_ERR_SHAPE, RL_ERR_DTYPE, RL_ERR_ALIGN, RL_ERR_ALIAS, \
    RL_ERR_WORKSPACE, RL_ERR_ID_RANGE, RL_ERR_TIMEOUT, RL_ERR_CUDA, RL_ERR_ARG = range(11)
RL_F32, RL_BF16, RL_F16 = 0, 1, 2
RL_ADV_PER_SEQ, RL_ADV_PER_TOKEN, RL_ADV_GROUP_REWARDS = 0, 1, 2
RL_AGG_TOKEN_MEAN, RL_AGG_SEQ_MEAN_TOKEN_MEAN, RL_AGG_SEQ_MEAN_TOKEN_SUM, RL_AGG_TOKEN_SUM_NORM = \
    0, 1, 2, 3
AGGREGATIONS = {"token_mean": 0, "seq_mean_token_mean": 1, "seq_mean_token_sum": 2,
                "token_sum_norm": 3}
RL_DEVERR_ID_RANGE, RL_DEVERR_TIMEOUT = 1, 2

DTYPES = {"f32": RL_F32, "bf16": RL_BF16, "f16": RL_F16}

__all__ = [
    "rl_group_advantages", "rl_gae_reverse_scan", "rl_policy_loss_workspace_size",
    "rl_policy_loss_fwd_bwd", "rl_policy_loss_fwd_bwd_ex", "rl_policy_loss_desc_init",
    "rl_policy_loss_desc", "rl_policy_loss_fwd_bwd_noalloc", "rl_policy_loss_launch_shape",
    "rl_read_device_status", "rl_masked_whiten", "rl_count_tokens", "rl_value_loss_fwd_bwd",
    "rl_value_stats", "value_stats_from_bytes", "rl_lmhead_logprobs",
    "rl_lmhead_workspace_size", "rl_lmhead_plan", "rl_selftest_wait_timeout",
    "rl_status_string", "rl_loss_stats", "RlLossError", "build", "load", "stats_from_bytes",
]


class RlLossError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {rl_status_string(status)} (status {status})")


class rl_loss_stats(ctypes.Structure):
    _fields_ = [("loss", ctypes.c_double), ("pg_term", ctypes.c_double),
                ("kl_term", ctypes.c_double), ("ent_term", ctypes.c_double),
                ("clip_frac", ctypes.c_double), ("n_tokens", ctypes.c_longlong),
                ("n_clipped", ctypes.c_longlong), ("device_error", ctypes.c_int),
                ("reserved", ctypes.c_int)]


class rl_policy_loss_desc(ctypes.Structure):
    _fields_ = [("logits", ctypes.c_void_p), ("dtype", ctypes.c_int),
                ("B", ctypes.c_longlong), ("T", ctypes.c_longlong), ("V", ctypes.c_longlong),
                ("ld", ctypes.c_longlong), ("ids", ctypes.c_void_p), ("logp_old", ctypes.c_void_p),
                ("ref_logp", ctypes.c_void_p), ("mask", ctypes.c_void_p), ("adv", ctypes.c_void_p),
                ("adv_layout", ctypes.c_int), ("group_size", ctypes.c_int), ("ddof", ctypes.c_int),
                ("std_eps", ctypes.c_double), ("eps", ctypes.c_float), ("eps_high", ctypes.c_float),
                ("beta", ctypes.c_float), ("c_ent", ctypes.c_float), ("grad_scale", ctypes.c_float),
                ("agg", ctypes.c_int), ("agg_norm", ctypes.c_double), ("dlogits", ctypes.c_void_p),
                ("logp_out", ctypes.c_void_p), ("entropy_out", ctypes.c_void_p),
                ("stats_dev", ctypes.c_void_p), ("workspace", ctypes.c_void_p),
                ("workspace_bytes", ctypes.c_size_t), ("global_counts", ctypes.c_void_p),
                ("vocab_offset", ctypes.c_longlong), ("vocab_total", ctypes.c_longlong),
                ("partials_out", ctypes.c_void_p), ("shard_partials", ctypes.c_void_p),
                ("n_shards", ctypes.c_int), ("row_coef_out", ctypes.c_void_p)]


class rl_value_stats(ctypes.Structure):
    _fields_ = [("loss", ctypes.c_double), ("clip_frac", ctypes.c_double),
                ("mean_abs_err", ctypes.c_double), ("n_tokens", ctypes.c_longlong),
                ("n_clipped", ctypes.c_longlong)]


STATS_BYTES = ctypes.sizeof(rl_loss_stats)
VALUE_STATS_BYTES = ctypes.sizeof(rl_value_stats)
_lib = None


def load(path: str | None = None):
    """Load librlloss.so (built in-tree by ``build()``); raises if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or LIB_PATH
    if not os.path.exists(path):
        raise RuntimeError(f"librlloss.so is not built ({path}); run ppo_policy_loss_gb300.build()")
    lib = ctypes.CDLL(path)
    P, LL, I, F, D, SZ = (ctypes.c_void_p, ctypes.c_longlong, ctypes.c_int, ctypes.c_float,
                          ctypes.c_double, ctypes.c_size_t)
    lib.rl_group_advantages.argtypes = [P, I, I, D, I, P, P]
    lib.rl_gae_reverse_scan.argtypes = [P, P, P, I, I, F, F, P, P, P]
    lib.rl_policy_loss_workspace_size.argtypes = [LL]
    lib.rl_policy_loss_workspace_size.restype = SZ
    lib.rl_policy_loss_fwd_bwd.argtypes = [P, I, LL, LL, LL, LL, P, P, P, P, P, I, F, F, F, F,
                                           P, P, P, P, P, SZ, P]
    lib.rl_policy_loss_fwd_bwd_noalloc.argtypes = [P, I, LL, LL, LL, LL, P, P, P, P, P, I, F, F,
                                                   F, F, P, P, P, P, P]
    lib.rl_policy_loss_desc_init.argtypes = [ctypes.POINTER(rl_policy_loss_desc)]
    lib.rl_policy_loss_desc_init.restype = None
    lib.rl_policy_loss_fwd_bwd_ex.argtypes = [ctypes.POINTER(rl_policy_loss_desc), P]
    lib.rl_value_loss_fwd_bwd.argtypes = [P, P, P, P, LL, F, F, P, P, P]
    lib.rl_masked_whiten.argtypes = [P, P, LL, D, I, P, P]
    lib.rl_count_tokens.argtypes = [P, LL, LL, P, P]
    lib.rl_lmhead_logprobs.argtypes = [P, LL, P, LL, I, LL, LL, LL, P, P, P, P, P, P, SZ, P]
    lib.rl_lmhead_workspace_size.argtypes = [LL, LL]
    lib.rl_lmhead_workspace_size.restype = SZ
    lib.rl_lmhead_plan.argtypes = [LL, LL, LL, SZ, I, ctypes.POINTER(I), ctypes.POINTER(I),
                                   ctypes.POINTER(I), ctypes.POINTER(SZ)]
    lib.rl_lmhead_plan.restype = I
    lib.rl_count_tokens.restype = I
    lib.rl_masked_whiten.restype = I
    lib.rl_lmhead_logprobs.restype = I
    lib.rl_lmhead_row_partials.argtypes = [P, LL, P, LL, I, LL, LL, LL, P, P, P, P, SZ, P]
    lib.rl_lmhead_dlogits.argtypes = [P, LL, P, LL, I, LL, LL, LL, P, P, P, LL, P, P]
    lib.rl_lmhead_dhidden.argtypes = [P, LL, P, LL, I, LL, LL, LL, P, LL, P, P]
    lib.rl_lmhead_dweight.argtypes = [P, LL, P, LL, I, LL, LL, LL, P, LL, I, P, P]
    for fn in ("rl_lmhead_row_partials", "rl_lmhead_dlogits", "rl_lmhead_dhidden",
               "rl_lmhead_dweight"):
        getattr(lib, fn).restype = I
    lib.rl_policy_loss_launch_shape.argtypes = [I, LL, LL, ctypes.POINTER(I), ctypes.POINTER(I),
                                                ctypes.POINTER(I)]
    lib.rl_read_device_status.argtypes = [P, P]
    lib.rl_selftest_wait_timeout.argtypes = [ctypes.c_ulonglong, P, P, P]
    lib.rl_selftest_wait_timeout.restype = I
    lib.rl_status_string.argtypes = [I]
    lib.rl_status_string.restype = ctypes.c_char_p
    for fn in ("rl_group_advantages", "rl_gae_reverse_scan", "rl_policy_loss_fwd_bwd",
               "rl_policy_loss_fwd_bwd_ex", "rl_policy_loss_fwd_bwd_noalloc", "rl_value_loss_fwd_bwd",
               "rl_policy_loss_launch_shape",
               "rl_read_device_status"):
        getattr(lib, fn).restype = I
    _lib = lib
    return lib


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _dtype(dt):
    return DTYPES[dt] if isinstance(dt, str) else int(dt)


def _check(status: int, where: str):
    if status != RL_OK:
        raise RlLossError(status, where)


def rl_status_string(status: int) -> str:
    return load().rl_status_string(int(status)).decode()


def rl_group_advantages(rewards, n_groups, group_size, std_eps, ddof, adv_out, stream=None):
    _check(load().rl_group_advantages(_ptr(rewards), n_groups, group_size, std_eps, ddof,
                                      _ptr(adv_out), _stream(stream)), "rl_group_advantages")


def rl_gae_reverse_scan(rewards, values, lengths, B, T, gamma, lam, adv_out, returns_out,
                        stream=None):
    _check(load().rl_gae_reverse_scan(_ptr(rewards), _ptr(values), _ptr(lengths), B, T, gamma, lam,
                                      _ptr(adv_out), _ptr(returns_out), _stream(stream)),
           "rl_gae_reverse_scan")


def rl_policy_loss_workspace_size(n_rows) -> int:
    return int(load().rl_policy_loss_workspace_size(n_rows))


def rl_policy_loss_fwd_bwd(logits, dtype, B, T, V, ld, ids, logp_old, ref_logp, mask, adv,
                           adv_layout, eps, beta, c_ent, grad_scale, dlogits, logp_out,
                           entropy_out, stats_dev, workspace, workspace_bytes, stream=None):
    _check(load().rl_policy_loss_fwd_bwd(
        _ptr(logits), _dtype(dtype), B, T, V, ld, _ptr(ids), _ptr(logp_old), _ptr(ref_logp),
        _ptr(mask), _ptr(adv), adv_layout, eps, beta, c_ent, grad_scale, _ptr(dlogits),
        _ptr(logp_out), _ptr(entropy_out), _ptr(stats_dev), _ptr(workspace), workspace_bytes,
        _stream(stream)), "rl_policy_loss_fwd_bwd")


def rl_policy_loss_desc_init() -> rl_policy_loss_desc:
    """A descriptor holding the library's defaults (see rl_policy_loss_desc_init)."""
    d = rl_policy_loss_desc()
    load().rl_policy_loss_desc_init(ctypes.byref(d))
    return d


def rl_policy_loss_fwd_bwd_ex(desc: rl_policy_loss_desc, stream=None):
    _check(load().rl_policy_loss_fwd_bwd_ex(ctypes.byref(desc), _stream(stream)),
           "rl_policy_loss_fwd_bwd_ex")


def rl_policy_loss_fwd_bwd_noalloc(logits, dtype, B, T, V, ld, ids, logp_old, ref_logp, mask,
                                   adv, adv_layout, eps, beta, c_ent, grad_scale, dlogits,
                                   logp_out, entropy_out, stats_dev, stream=None):
    """rl_policy_loss_fwd_bwd with the library's own static scratch instead of a
    caller workspace, for callers that cannot allocate device memory.  Calls
    share that scratch: do not let two of them overlap on the GPU."""
    _check(load().rl_policy_loss_fwd_bwd_noalloc(
        _ptr(logits), _dtype(dtype), B, T, V, ld, _ptr(ids), _ptr(logp_old), _ptr(ref_logp),
        _ptr(mask), _ptr(adv), adv_layout, eps, beta, c_ent, grad_scale, _ptr(dlogits),
        _ptr(logp_out), _ptr(entropy_out), _ptr(stats_dev), _stream(stream)),
        "rl_policy_loss_fwd_bwd_noalloc")


def rl_value_loss_fwd_bwd(values, values_old, returns, mask, n, clip_eps, grad_scale, dvalues,
                          stats_dev, stream=None):
    _check(load().rl_value_loss_fwd_bwd(_ptr(values), _ptr(values_old), _ptr(returns), _ptr(mask),
                                        n, clip_eps, grad_scale, _ptr(dvalues), _ptr(stats_dev),
                                        _stream(stream)), "rl_value_loss_fwd_bwd")


def rl_masked_whiten(x, mask, n, eps, shift_mean, out, stream=None):
    _check(load().rl_masked_whiten(_ptr(x), _ptr(mask), n, eps, int(shift_mean), _ptr(out),
                                   _stream(stream)), "rl_masked_whiten")


def rl_count_tokens(mask, B, T, counts_dev, stream=None):
    _check(load().rl_count_tokens(_ptr(mask), B, T, _ptr(counts_dev), _stream(stream)),
           "rl_count_tokens")


def value_stats_from_bytes(raw: bytes) -> dict:
    """Decode a host copy of one rl_value_stats record."""
    st = rl_value_stats.from_buffer_copy(bytes(raw))
    return {name: getattr(st, name) for name, _ in rl_value_stats._fields_}


def rl_lmhead_logprobs(hidden, ld_h, weight, ld_w, dtype, R, D, V, ids, logp_out, entropy_out,
                       lse_out, status_dev=None, workspace=None, workspace_bytes=0, stream=None):
    if workspace is not None and hasattr(workspace, "numel") and not workspace_bytes:
        workspace_bytes = workspace.numel() * workspace.element_size()
    _check(load().rl_lmhead_logprobs(_ptr(hidden), ld_h, _ptr(weight), ld_w, _dtype(dtype), R, D, V,
                                     _ptr(ids), _ptr(logp_out), _ptr(entropy_out), _ptr(lse_out),
                                     _ptr(status_dev), _ptr(workspace), workspace_bytes,
                                     _stream(stream)), "rl_lmhead_logprobs")


def rl_lmhead_row_partials(hidden, ld_h, weight, ld_w, dtype, R, D, V, ids, partials_out,
                           status_dev=None, workspace=None, workspace_bytes=0, stream=None):
    if workspace is not None and hasattr(workspace, "numel") and not workspace_bytes:
        workspace_bytes = workspace.numel() * workspace.element_size()
    _check(load().rl_lmhead_row_partials(_ptr(hidden), ld_h, _ptr(weight), ld_w, _dtype(dtype), R, D,
                                         V, _ptr(ids), _ptr(partials_out), _ptr(status_dev),
                                         _ptr(workspace), workspace_bytes, _stream(stream)),
           "rl_lmhead_row_partials")


def rl_lmhead_dlogits(hidden, ld_h, weight, ld_w, dtype, R, D, V, ids, row_coef, dlogits, ld_dz,
                      status_dev=None, stream=None):
    _check(load().rl_lmhead_dlogits(_ptr(hidden), ld_h, _ptr(weight), ld_w, _dtype(dtype), R, D, V,
                                    _ptr(ids), _ptr(row_coef), _ptr(dlogits), ld_dz,
                                    _ptr(status_dev), _stream(stream)), "rl_lmhead_dlogits")


def rl_lmhead_dhidden(dlogits, ld_dz, weight, ld_w, dtype, R, D, V, dhidden, ld_dh,
                      status_dev=None, stream=None):
    _check(load().rl_lmhead_dhidden(_ptr(dlogits), ld_dz, _ptr(weight), ld_w, _dtype(dtype), R, D, V,
                                    _ptr(dhidden), ld_dh, _ptr(status_dev), _stream(stream)),
           "rl_lmhead_dhidden")


def rl_lmhead_dweight(dlogits, ld_dz, hidden, ld_h, dtype, R, D, V, dweight, ld_dw, accumulate,
                      status_dev=None, stream=None):
    _check(load().rl_lmhead_dweight(_ptr(dlogits), ld_dz, _ptr(hidden), ld_h, _dtype(dtype), R, D, V,
                                    _ptr(dweight), ld_dw, int(accumulate), _ptr(status_dev),
                                    _stream(stream)), "rl_lmhead_dweight")


def rl_lmhead_workspace_size(R, V) -> int:
    return int(load().rl_lmhead_workspace_size(R, V))


def rl_lmhead_plan(R, D, V, workspace_bytes, sm_count=0):
    """(vocabulary slices per row tile, CTAs, row tiles per unit group, workspace
    bytes used) of the launch on a GPU of ``sm_count`` SMs (0: the current
    device); the C call's outputs in their order."""
    ns, grid, grp, need = ctypes.c_int(0), ctypes.c_int(0), ctypes.c_int(0), ctypes.c_size_t(0)
    _check(load().rl_lmhead_plan(R, D, V, workspace_bytes, sm_count, ctypes.byref(ns),
                                 ctypes.byref(grid), ctypes.byref(grp), ctypes.byref(need)),
           "rl_lmhead_plan")
    return ns.value, grid.value, grp.value, need.value


def rl_policy_loss_launch_shape(dtype, V, n_rows):
    c, n, s = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
    _check(load().rl_policy_loss_launch_shape(_dtype(dtype), V, n_rows, ctypes.byref(c),
                                              ctypes.byref(n), ctypes.byref(s)),
           "rl_policy_loss_launch_shape")
    return c.value, n.value, s.value


def rl_selftest_wait_timeout(limit_ns, status_dev, waited_ns_dev=None, stream=None):
    _check(load().rl_selftest_wait_timeout(int(limit_ns), _ptr(status_dev), _ptr(waited_ns_dev),
                                           _stream(stream)), "rl_selftest_wait_timeout")


def rl_read_device_status(workspace, stream=None) -> int:
    """Synchronises the stream; returns the status code (does not raise)."""
    return int(load().rl_read_device_status(_ptr(workspace), _stream(stream)))


def stats_from_bytes(raw: bytes) -> dict:
    """Decode a host copy of one rl_loss_stats record."""
    st = rl_loss_stats.from_buffer_copy(bytes(raw))
    return {name: getattr(st, name) for name, _ in rl_loss_stats._fields_}
