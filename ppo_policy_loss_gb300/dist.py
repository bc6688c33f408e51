"""Data parallelism over ranks for the fused policy loss.

Rows are independent, so a batch shards by whole sequences (whole GRPO
groups) with no exchange on the data path except the token counts: the
global token mean needs N (and B' for the sequence-level aggregations)
summed over ranks before the loss kernel runs, and the loss is the sum of
the ranks' shares after.  That is two all-reduces of 16 and 8 bytes; the
gradient of each rank's logits stays on its GPU.

torch.distributed is the transport (NCCL on GPUs, gloo in the CPU tests);
every computation runs in the library's kernels.  ``count_fn`` and
``loss_fn`` exist so the orchestration can be exercised without a GPU.
"""
from __future__ import annotations

import torch
import torch.distributed as dist

from . import torch_api


def _default_loss(logits, ids, mask, adv, B, T, global_counts, **kw):
    out = torch_api.policy_loss(logits, ids, mask, adv, B, T, global_counts=global_counts, **kw)
    out["loss_share"] = out["stats"][:8].view(torch.float64).clone()
    return out


def policy_loss_data_parallel(logits, ids, mask, adv, B, T, group=None, count_fn=None,
                              loss_fn=None, **kw) -> dict:
    """Fused loss of this rank's rows, normalised over every rank's tokens.

    Returns the outputs of ``torch_api.policy_loss`` plus ``global_counts``
    (int64[2]: N, B' over all ranks) and ``loss`` (float64[1]: the global
    loss, the same on every rank).  Collectives are issued on the current
    stream's device in the same order on every rank.
    """
    count_fn = count_fn or (lambda m, b, t: torch_api.count_tokens(m, b, t))
    loss_fn = loss_fn or _default_loss
    counts = count_fn(mask, B, T)
    dist.all_reduce(counts, op=dist.ReduceOp.SUM, group=group)
    out = loss_fn(logits, ids, mask, adv, B, T, counts, **kw)
    share = out["loss_share"]
    dist.all_reduce(share, op=dist.ReduceOp.SUM, group=group)
    out["global_counts"] = counts
    out["loss"] = share
    return out
