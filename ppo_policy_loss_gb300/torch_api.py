"""Convenience layer over the C ABI for callers that hold torch CUDA tensors.

It only allocates outputs with torch (device memory) and forwards to the C
entry points; every step of the computation runs in librlloss's kernels.
"""
from __future__ import annotations

import torch

from . import (AGGREGATIONS, DTYPES, RL_ADV_GROUP_REWARDS, RL_ADV_PER_SEQ, RL_ADV_PER_TOKEN,
               STATS_BYTES, rl_gae_reverse_scan, rl_group_advantages, rl_policy_loss_desc_init,
               VALUE_STATS_BYTES, rl_count_tokens, rl_lmhead_logprobs, rl_lmhead_workspace_size,
               rl_masked_whiten, rl_policy_loss_fwd_bwd_ex, rl_policy_loss_workspace_size,
               rl_value_loss_fwd_bwd, stats_from_bytes, value_stats_from_bytes)

_DT = {torch.float32: "f32", torch.bfloat16: "bf16", torch.float16: "f16"}


def dtype_name(t: torch.Tensor) -> str:
    return _DT[t.dtype]


def new_workspace(n_rows: int, device) -> torch.Tensor:
    """Zero-filled workspace (the library leaves it ready for reuse after each call)."""
    return torch.zeros(rl_policy_loss_workspace_size(n_rows), dtype=torch.uint8, device=device)


def new_stats(device) -> torch.Tensor:
    return torch.zeros(STATS_BYTES, dtype=torch.uint8, device=device)


def read_stats(stats: torch.Tensor) -> dict:
    return stats_from_bytes(stats.cpu().numpy().tobytes())


def group_advantages(rewards: torch.Tensor, group_size: int, std_eps: float = 1e-4,
                     ddof: int = 1, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    out = torch.empty_like(rewards) if out is None else out
    n = rewards.numel()
    rl_group_advantages(rewards, n // group_size, group_size, std_eps, ddof, out, stream)
    return out


def gae(rewards: torch.Tensor, values: torch.Tensor, lengths: torch.Tensor, gamma: float,
        lam: float, want_returns: bool = True, stream=None):
    B, T = rewards.shape
    adv = torch.empty_like(rewards)
    ret = torch.empty_like(rewards) if want_returns else None
    rl_gae_reverse_scan(rewards, values, lengths, B, T, gamma, lam, adv, ret, stream)
    return adv, ret


def policy_loss(logits: torch.Tensor, ids: torch.Tensor, mask: torch.Tensor, adv: torch.Tensor,
                B: int, T: int, V: int | None = None, logp_old=None, ref_logp=None,
                eps: float = 0.2, beta: float = 0.0, c_ent: float = 0.0, grad_scale: float = 1.0,
                dlogits="new", logp_out="new", entropy_out="new", workspace=None, stats=None,
                stream=None, eps_high: float | None = None, agg: str = "token_mean",
                agg_norm: float = 1.0, group_size: int | None = None, ddof: int = 1,
                std_eps: float = 1e-4, global_counts: torch.Tensor | None = None,
                vocab_offset: int = 0, vocab_total: int = 0, partials_out=None,
                shard_partials=None) -> dict:
    """Run the fused loss on [B*T, ld] logits (rl_policy_loss_fwd_bwd_ex).

    ``dlogits`` / ``logp_out`` / ``entropy_out``: "new" allocates, None skips,
    a tensor is written in place (``dlogits=logits`` is the in-place form).
    ``adv`` of B elements is per sequence, of B*T elements per token; with
    ``group_size`` set, ``adv`` holds the B rewards and the launch computes the
    group-relative advantages itself.  ``agg`` names the loss aggregation
    (token_mean, seq_mean_token_mean, seq_mean_token_sum, token_sum_norm).
    Returns the output tensors and the (device) stats record; call
    ``read_stats`` for the scalars.

    Vocabulary shards: ``logits`` holds columns [vocab_offset, vocab_offset + V)
    of a ``vocab_total``-column vocabulary.  With ``partials_out`` (float32
    [B*T, 4]) the launch only writes each row's shard statistics; with
    ``shard_partials`` (float32 [n_shards, B*T, 4], every shard's partials in
    shard order) it merges them and computes the loss and this shard's
    gradient columns.
    """
    dev = logits.device
    R = B * T
    if partials_out is not None:  # this launch writes the shard partials only
        dlogits = logp_out = entropy_out = None
    ld = logits.stride(0) if logits.dim() == 2 and R > 0 else logits.shape[-1]
    V = logits.shape[-1] if V is None else V
    if isinstance(dlogits, str):  # same row stride as the logits (the C call takes one ld)
        if logits.dim() == 2 and logits.stride(0) != logits.shape[1]:
            dlogits = torch.empty((logits.shape[0], ld), dtype=logits.dtype, device=dev)
            dlogits = dlogits[:, :logits.shape[1]]
        else:
            dlogits = torch.empty_like(logits)
    elif dlogits is not None and R > 0 and dlogits.stride(0) != ld:
        raise ValueError(f"dlogits row stride {dlogits.stride(0)} != logits row stride {ld}")
    if isinstance(logp_out, str):
        logp_out = torch.empty(R, dtype=torch.float32, device=dev)
    if isinstance(entropy_out, str):
        entropy_out = torch.empty(R, dtype=torch.float32, device=dev)
    workspace = new_workspace(R, dev) if workspace is None else workspace
    stats = new_stats(dev) if stats is None else stats
    if group_size is not None:
        layout = RL_ADV_GROUP_REWARDS
    else:
        layout = RL_ADV_PER_TOKEN if adv.numel() == R and R != B else RL_ADV_PER_SEQ
    d = rl_policy_loss_desc_init()
    p = lambda t: t.data_ptr() if t is not None else None
    d.logits, d.dtype, d.B, d.T, d.V, d.ld = p(logits), DTYPES[dtype_name(logits)], B, T, V, ld
    d.ids, d.logp_old, d.ref_logp, d.mask, d.adv = p(ids), p(logp_old), p(ref_logp), p(mask), p(adv)
    d.adv_layout = layout
    if group_size is not None:
        d.group_size, d.ddof, d.std_eps = group_size, ddof, std_eps
    d.eps, d.eps_high = eps, (-1.0 if eps_high is None else eps_high)
    d.beta, d.c_ent, d.grad_scale = beta, c_ent, grad_scale
    d.agg, d.agg_norm = AGGREGATIONS[agg], agg_norm
    d.dlogits, d.logp_out, d.entropy_out = p(dlogits), p(logp_out), p(entropy_out)
    d.stats_dev, d.workspace, d.workspace_bytes = p(stats), p(workspace), workspace.numel()
    d.global_counts = p(global_counts)
    d.vocab_offset, d.vocab_total = vocab_offset, vocab_total
    d.partials_out, d.shard_partials = p(partials_out), p(shard_partials)
    d.n_shards = shard_partials.shape[0] if shard_partials is not None else 0
    rl_policy_loss_fwd_bwd_ex(d, stream)
    return dict(dlogits=dlogits, logp=logp_out, entropy=entropy_out, stats=stats,
                workspace=workspace)


def policy_loss_from_partials(partials: torch.Tensor, dtype: str, vocab: int, ids: torch.Tensor,
                              mask: torch.Tensor, adv: torch.Tensor, B: int, T: int, logp_old=None,
                              ref_logp=None, eps: float = 0.2, beta: float = 0.0, c_ent: float = 0.0,
                              grad_scale: float = 1.0, logp_out="new", entropy_out="new",
                              workspace=None, stats=None, stream=None,
                              eps_high: float | None = None, agg: str = "token_mean",
                              agg_norm: float = 1.0, group_size: int | None = None, ddof: int = 1,
                              std_eps: float = 1e-4,
                              global_counts: torch.Tensor | None = None) -> dict:
    """The loss, its statistics, logp, entropy and each row's gradient
    coefficients from per-row softmax statistics of a ``vocab``-column
    vocabulary, without any logits: the merge launch of
    rl_policy_loss_fwd_bwd_ex with no columns of its own (V = 0) and
    ``row_coef_out``.  ``partials`` is float32 [B*T, 4] (one shard, e.g. from
    rl_lmhead_row_partials) or [n_shards, B*T, 4]; ``dtype`` names the
    16-bit format the gradient will be formed in.  Returns the outputs and
    ``row_coef`` float32 [B*T, 4] (cL, a0, a1, gy) for rl_lmhead_dlogits."""
    dev = partials.device
    R = B * T
    if partials.dim() == 2:
        partials = partials[None]
    if isinstance(logp_out, str):
        logp_out = torch.empty(R, dtype=torch.float32, device=dev)
    if isinstance(entropy_out, str):
        entropy_out = torch.empty(R, dtype=torch.float32, device=dev)
    coef = torch.empty((R, 4), dtype=torch.float32, device=dev)
    workspace = new_workspace(R, dev) if workspace is None else workspace
    stats = new_stats(dev) if stats is None else stats
    if group_size is not None:
        layout = RL_ADV_GROUP_REWARDS
    else:
        layout = RL_ADV_PER_TOKEN if adv.numel() == R and R != B else RL_ADV_PER_SEQ
    d = rl_policy_loss_desc_init()
    p = lambda t: t.data_ptr() if t is not None else None
    d.logits, d.dtype, d.B, d.T, d.V, d.ld = None, DTYPES[dtype], B, T, 0, 0
    d.ids, d.logp_old, d.ref_logp, d.mask, d.adv = p(ids), p(logp_old), p(ref_logp), p(mask), p(adv)
    d.adv_layout = layout
    if group_size is not None:
        d.group_size, d.ddof, d.std_eps = group_size, ddof, std_eps
    d.eps, d.eps_high = eps, (-1.0 if eps_high is None else eps_high)
    d.beta, d.c_ent, d.grad_scale = beta, c_ent, grad_scale
    d.agg, d.agg_norm = AGGREGATIONS[agg], agg_norm
    d.dlogits, d.logp_out, d.entropy_out = None, p(logp_out), p(entropy_out)
    d.stats_dev, d.workspace, d.workspace_bytes = p(stats), p(workspace), workspace.numel()
    d.global_counts = p(global_counts)
    d.vocab_offset, d.vocab_total = 0, vocab
    d.shard_partials, d.n_shards = p(partials), partials.shape[0]
    d.row_coef_out = p(coef)
    rl_policy_loss_fwd_bwd_ex(d, stream)
    return dict(logp=logp_out, entropy=entropy_out, stats=stats, row_coef=coef, workspace=workspace)


def value_loss(values: torch.Tensor, returns: torch.Tensor, mask: torch.Tensor, values_old=None,
               clip_eps: float = -1.0, grad_scale: float = 1.0, dvalues="new", stream=None):
    """PPO clipped value loss (rl_value_loss_fwd_bwd); returns (dvalues, stats dict)."""
    n = values.numel()
    if isinstance(dvalues, str):
        dvalues = torch.empty_like(values)
    st = torch.zeros(VALUE_STATS_BYTES, dtype=torch.uint8, device=values.device)
    rl_value_loss_fwd_bwd(values, values_old, returns, mask, n, clip_eps, grad_scale, dvalues, st,
                          stream)
    return dvalues, value_stats_from_bytes(st.cpu().numpy().tobytes())


class FusedPolicyLoss(torch.autograd.Function):
    """Autograd wrapper: forward runs the fused kernel once and keeps its
    logits gradient; backward hands that gradient back, scaled by the
    incoming gradient (a no-op when it is exactly 1, the usual case).

    loss = FusedPolicyLoss.apply(logits, ids, mask, adv, B, T, options)
    with ``options`` a dict of policy_loss keyword arguments (logp_old,
    ref_logp, eps, beta, c_ent, eps_high, agg, agg_norm, group_size, ...).
    ``options["inplace"] = True`` writes the gradient over the logits
    (saves one logits-sized buffer; the logits are then gone).
    """

    @staticmethod
    def forward(ctx, logits, ids, mask, adv, B, T, options=None):
        opts = dict(options or {})
        inplace = opts.pop("inplace", False)
        out = policy_loss(logits.detach(), ids, mask, adv, B, T,
                          dlogits=logits.detach() if inplace else "new", **opts)
        ctx.save_for_backward(out["dlogits"])
        ctx.stats = out["stats"]
        ctx.mark_non_differentiable(out["logp"], out["entropy"])
        loss = out["stats"][:8].view(torch.float64)[0].clone()
        return loss, out["logp"], out["entropy"]

    @staticmethod
    def backward(ctx, grad_loss, _g_logp, _g_ent):
        (dlogits,) = ctx.saved_tensors
        if grad_loss is not None and float(grad_loss) != 1.0:
            dlogits = dlogits * grad_loss.to(dlogits.dtype)
        return dlogits, None, None, None, None, None, None


def masked_whiten(x: torch.Tensor, mask: torch.Tensor, eps: float = 1e-8, shift_mean: bool = True,
                  out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Masked advantage whitening (rl_masked_whiten)."""
    out = torch.empty_like(x) if out is None else out
    rl_masked_whiten(x, mask, x.numel(), eps, shift_mean, out, stream)
    return out


def count_tokens(mask: torch.Tensor, B: int, T: int, out: torch.Tensor | None = None,
                 stream=None) -> torch.Tensor:
    """Device int64[2] = (N, B') of the batch (rl_count_tokens)."""
    out = torch.empty(2, dtype=torch.int64, device=mask.device) if out is None else out
    rl_count_tokens(mask, B, T, out, stream)
    return out


def lmhead_logprobs(hidden: torch.Tensor, weight: torch.Tensor, ids: torch.Tensor,
                    want_entropy: bool = True, want_lse: bool = False, workspace="new",
                    status: torch.Tensor | None = None, stream=None) -> dict:
    """Per-row log-probs of the sampled ids (and entropy, lse) of hidden @ weight.T
    without forming the logits (rl_lmhead_logprobs).  hidden [R, D] and weight
    [V, D] are bf16 or fp16 CUDA tensors (the same type) with unit column stride.  ``workspace``: "new"
    allocates the size the launch can use to balance the SMs, None runs
    unsliced, a uint8 tensor is used as given (zero-filled before first use)."""
    R, D = hidden.shape
    V = weight.shape[0]
    dev = hidden.device
    logp = torch.empty(R, dtype=torch.float32, device=dev)
    ent = torch.empty(R, dtype=torch.float32, device=dev) if want_entropy else None
    lse = torch.empty(R, dtype=torch.float32, device=dev) if want_lse else None
    if isinstance(workspace, str):
        nb = rl_lmhead_workspace_size(R, V)
        workspace = torch.zeros(nb, dtype=torch.uint8, device=dev) if nb else None
    rl_lmhead_logprobs(hidden, hidden.stride(0), weight, weight.stride(0), dtype_name(hidden), R, D, V,
                       ids, logp, ent,
                       lse, status, workspace, workspace.numel() if workspace is not None else 0,
                       stream)
    return dict(logp=logp, entropy=ent, lse=lse, workspace=workspace)
