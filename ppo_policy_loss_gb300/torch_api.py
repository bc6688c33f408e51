"""Convenience layer over the C ABI for callers that hold torch CUDA tensors.

It only allocates outputs with torch (device memory) and forwards to the C
entry points; every step of the computation runs in librlloss's kernels.
"""
from __future__ import annotations

import torch

from . import (RL_ADV_PER_SEQ, RL_ADV_PER_TOKEN, STATS_BYTES, rl_gae_reverse_scan,
               rl_group_advantages, rl_policy_loss_fwd_bwd, rl_policy_loss_workspace_size,
               stats_from_bytes)

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
                stream=None) -> dict:
    """Run rl_policy_loss_fwd_bwd on [B*T, ld] logits.

    ``dlogits`` / ``logp_out`` / ``entropy_out``: "new" allocates, None skips,
    a tensor is written in place (``dlogits=logits`` is the in-place form).
    ``adv`` of B elements is per sequence, of B*T elements per token.
    Returns the output tensors and the (device) stats record; call
    ``read_stats`` for the scalars.
    """
    dev = logits.device
    R = B * T
    ld = logits.stride(0) if logits.dim() == 2 and R > 0 else logits.shape[-1]
    V = logits.shape[-1] if V is None else V
    if isinstance(dlogits, str):
        dlogits = torch.empty_like(logits)
    if isinstance(logp_out, str):
        logp_out = torch.empty(R, dtype=torch.float32, device=dev)
    if isinstance(entropy_out, str):
        entropy_out = torch.empty(R, dtype=torch.float32, device=dev)
    workspace = new_workspace(R, dev) if workspace is None else workspace
    stats = new_stats(dev) if stats is None else stats
    layout = RL_ADV_PER_TOKEN if adv.numel() == R and R != B else RL_ADV_PER_SEQ
    rl_policy_loss_fwd_bwd(logits, dtype_name(logits), B, T, V, ld, ids, logp_old, ref_logp, mask,
                           adv, layout, eps, beta, c_ent, grad_scale, dlogits, logp_out,
                           entropy_out, stats, workspace, workspace.numel(), stream)
    return dict(dlogits=dlogits, logp=logp_out, entropy=entropy_out, stats=stats,
                workspace=workspace)
