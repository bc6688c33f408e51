"""The policy loss from hidden states, forward and backward, with the logits
never in HBM.

The actor's logits are its LM-head output z = hidden @ W^T (ainews.cool RL.cu
article, section "技术深度解析", policy and value networks bullet: the actor's
own matrix multiplications, 16-bit inputs with fp32 accumulation per the
pitchhut.com RL.cu listing, "Key Features" item 1).  Every step below is one
of this library's kernels, called through its C ABI:

  1. rl_lmhead_row_partials: z tile by tile on the tensor cores, folded into
     each row's softmax statistics (max, sum 2^x, sum 2^x x, sampled logit);
  2. rl_policy_loss_fwd_bwd_ex, merge launch with no columns: the loss, its
     statistics, logp, entropy and each row's gradient coefficients, for the
     whole batch in one launch;
  3. per chunk of sequences:
       rl_lmhead_dlogits: z recomputed on the tensor cores and turned into
         the loss gradient dz in the epilogue (the only R x V array written);
       rl_lmhead_dhidden: dhidden = dz @ W;
       rl_lmhead_dweight: dW (+)= dz^T @ hidden, fp32.

The forward statistics and the gradient each form z once: four R x D x V
products in all, against three for a chain that writes the logits and reads
them back.  Peak extra memory is one chunk of dz (``chunk_bytes``).
"""
from __future__ import annotations

import torch

from . import (rl_lmhead_dhidden, rl_lmhead_dlogits, rl_lmhead_dweight, rl_lmhead_row_partials,
               rl_lmhead_workspace_size, torch_api)


def _seqs_per_chunk(B: int, T: int, V: int, elem: int, chunk_bytes: int) -> int:
    return max(1, min(B, chunk_bytes // max(1, T * V * elem)))


def lmhead_policy_loss(hidden: torch.Tensor, weight: torch.Tensor, ids: torch.Tensor,
                       mask: torch.Tensor, adv: torch.Tensor, B: int, T: int,
                       chunk_bytes: int = 16 << 30, seqs_per_chunk: int | None = None,
                       stream=None, **loss_kw) -> dict:
    """Loss, statistics and the gradients with respect to ``hidden`` [B*T, D]
    and ``weight`` [V, D] (bf16 or fp16 CUDA tensors, the same type, unit
    column stride) of the fused policy loss on the logits hidden @ weight^T.
    ``adv`` holds B per-sequence advantages, B*T per-token ones, or (with
    ``group_size`` in ``loss_kw``) the B rewards.  ``loss_kw`` are the
    torch_api.policy_loss options (logp_old, ref_logp, eps, beta, c_ent,
    eps_high, agg, agg_norm, grad_scale, group_size, ...); logp_old and
    ref_logp are per-token [B*T] tensors.

    Returns dict(loss: float64[1] device tensor, stats: float64[5] device
    tensor (loss, pg, kl, entropy, clip fraction), n_tokens: int64[1] device
    tensor, logp, entropy: float32[B*T], dhidden: like hidden, dweight:
    float32 [V, D], seqs_per_chunk, status: int32[1] device error bits of the
    LM-head kernels)."""
    R, D = hidden.shape
    V = weight.shape[0]
    assert R == B * T and weight.shape[1] == D and weight.dtype == hidden.dtype
    dt = torch_api.dtype_name(hidden)
    dev = hidden.device
    ld_h, ld_w = hidden.stride(0), weight.stride(0)
    S = seqs_per_chunk or _seqs_per_chunk(B, T, V, hidden.element_size(), chunk_bytes)
    status = torch.zeros(1, dtype=torch.int32, device=dev)

    # 1. each row's softmax statistics of hidden @ W^T, the logits never written
    parts = torch.empty((R, 4), dtype=torch.float32, device=dev)
    nb = rl_lmhead_workspace_size(R, V)
    ws = torch.zeros(nb, dtype=torch.uint8, device=dev) if nb else None
    rl_lmhead_row_partials(hidden, ld_h, weight, ld_w, dt, R, D, V, ids, parts, status, ws,
                           nb, stream)
    # 2. the loss of the whole batch and each row's gradient coefficients
    out = torch_api.policy_loss_from_partials(parts, dt, V, ids, mask, adv, B, T, stream=stream,
                                              **loss_kw)
    coef = out["row_coef"]
    # 3. per chunk of sequences: dz from the hidden states, then both products
    dz = torch.empty((min(S, B) * T, V), dtype=hidden.dtype, device=dev)
    dhidden = torch.empty_like(hidden)
    dweight = torch.empty((V, D), dtype=torch.float32, device=dev)
    for b0 in range(0, B, S):
        r0, r1 = b0 * T, min(B, b0 + S) * T
        rows = r1 - r0
        rl_lmhead_dlogits(hidden[r0:r1], ld_h, weight, ld_w, dt, rows, D, V, ids[r0:r1],
                          coef[r0:r1], dz, V, status, stream)
        rl_lmhead_dhidden(dz, V, weight, ld_w, dt, rows, D, V, dhidden[r0:r1], D, status, stream)
        rl_lmhead_dweight(dz, V, hidden[r0:r1], ld_h, dt, rows, D, V, dweight, D, b0 > 0, status,
                          stream)
    st = out["stats"]
    stats = st[:40].view(torch.float64)
    return dict(loss=stats[:1].clone(), stats=stats, n_tokens=st[40:48].view(torch.int64),
                logp=out["logp"], entropy=out["entropy"], dhidden=dhidden, dweight=dweight,
                seqs_per_chunk=S, status=status, loss_stats=st)


class LMHeadPolicyLoss(torch.autograd.Function):
    """Autograd wrapper: forward runs lmhead_policy_loss and keeps its
    gradients; backward hands them back scaled by the incoming gradient.

    loss = LMHeadPolicyLoss.apply(hidden, weight, ids, mask, adv, B, T, options)
    """

    @staticmethod
    def forward(ctx, hidden, weight, ids, mask, adv, B, T, options=None):
        out = lmhead_policy_loss(hidden.detach(), weight.detach(), ids, mask, adv, B, T,
                                 **dict(options or {}))
        ctx.save_for_backward(out["dhidden"], out["dweight"])
        ctx.weight_dtype = weight.dtype
        return out["loss"][0].clone()

    @staticmethod
    def backward(ctx, grad):
        dh, dw = ctx.saved_tensors
        if grad is not None and float(grad) != 1.0:
            dh = dh * grad.to(dh.dtype)
            dw = dw * grad.to(dw.dtype)
        return dh, dw.to(ctx.weight_dtype), None, None, None, None, None, None
