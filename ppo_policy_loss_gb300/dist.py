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


def _default_partials(logits, ids, mask, adv, B, T, vocab_offset, vocab_total, **kw):
    R = B * T
    part = torch.empty((R, 4), dtype=torch.float32, device=logits.device)
    torch_api.policy_loss(logits, ids, mask, adv, B, T, vocab_offset=vocab_offset,
                          vocab_total=vocab_total, partials_out=part, **kw)
    return part


def _default_merge(logits, ids, mask, adv, B, T, vocab_offset, vocab_total, gathered, **kw):
    return torch_api.policy_loss(logits, ids, mask, adv, B, T, vocab_offset=vocab_offset,
                                 vocab_total=vocab_total, shard_partials=gathered, **kw)


def policy_loss_vocab_parallel(logits, ids, mask, adv, B, T, vocab_offset, vocab_total,
                               group=None, partials_fn=None, merge_fn=None, **kw) -> dict:
    """Fused loss with the vocabulary split over the ranks of ``group`` (each
    holds the logits columns [vocab_offset, vocab_offset + V) of every row; ids
    are global).  One launch per rank writes each row's shard statistics
    (max, sum of exponentials, their weighted sum, the sampled logit or -inf),
    an all-gather assembles them in rank order (B*T*16 bytes per rank), and a
    second launch merges them and writes the loss, logp, entropy and this
    rank's gradient columns.  Every rank reports the same loss."""
    partials_fn = partials_fn or _default_partials
    merge_fn = merge_fn or _default_merge
    part = partials_fn(logits, ids, mask, adv, B, T, vocab_offset, vocab_total, **kw)
    world = dist.get_world_size(group)
    flat = torch.empty((world * part.shape[0],) + tuple(part.shape[1:]), dtype=part.dtype,
                       device=part.device)
    dist.all_gather_into_tensor(flat, part.contiguous(), group=group)
    gathered = flat.view((world,) + tuple(part.shape))
    return merge_fn(logits, ids, mask, adv, B, T, vocab_offset, vocab_total, gathered, **kw)
