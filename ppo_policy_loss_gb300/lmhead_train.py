"""The policy loss from hidden states, forward and backward, in chunks of
whole sequences.

For each chunk of sequences:
  1. logits = hidden_c @ W^T            (library bf16 GEMM, into one reused buffer)
  2. the fused loss kernel reads those logits and writes dlogits over them in
     place, normalised by the token counts of the WHOLE batch
     (rl_count_tokens once, then ``global_counts``), so the chunks' loss
     shares add up to the batch loss;
  3. dhidden_c = dlogits @ W and dW += dlogits^T @ hidden_c   (library GEMMs;
     dW accumulated in fp32 across chunks).

The logits of the whole batch never exist at once: peak extra memory is one
chunk of logits (``chunk_bytes``, default 2 GiB) instead of B*T*V elements
(10 GB at 32 x 1024 x 151936 bf16).  The GEMMs are plain library GEMMs; the
loss, its gradient and the token counts run in this library's kernels.
"""
from __future__ import annotations

import torch

from . import torch_api


_ADDMM_F32 = [None]  # does torch.addmm take out_dtype (fp32 accumulation into a fp32 buffer)?


def _accumulate_f32(acc: torch.Tensor, a: torch.Tensor, b: torch.Tensor) -> None:
    """acc (fp32) += a @ b for bf16 a, b: one library GEMM with beta = 1 where
    the installed torch exposes an fp32 output for bf16 inputs, else a bf16
    product added in fp32."""
    if _ADDMM_F32[0] is not False:
        try:
            torch.addmm(acc, a, b, out_dtype=torch.float32, out=acc)
            _ADDMM_F32[0] = True
            return
        except (TypeError, RuntimeError):
            _ADDMM_F32[0] = False
    acc += torch.matmul(a, b).float()


def _seqs_per_chunk(B: int, T: int, V: int, elem: int, group: int, chunk_bytes: int) -> int:
    s = max(1, chunk_bytes // max(1, T * V * elem))
    s = max(group, s // group * group)  # whole groups: advantages may be computed in the launch
    return min(B, s)


def lmhead_policy_loss(hidden: torch.Tensor, weight: torch.Tensor, ids: torch.Tensor,
                       mask: torch.Tensor, adv: torch.Tensor, B: int, T: int,
                       chunk_bytes: int = 2 << 30, seqs_per_chunk: int | None = None,
                       **loss_kw) -> dict:
    """Loss, statistics and the gradients with respect to ``hidden`` [B*T, D]
    and ``weight`` [V, D] (both bf16 CUDA tensors) of the fused policy loss on
    the logits hidden @ weight^T.  ``adv`` holds B per-sequence advantages,
    B*T per-token ones, or (with ``group_size`` in ``loss_kw``) the B rewards.
    ``loss_kw`` are torch_api.policy_loss options (logp_old, ref_logp, eps,
    beta, c_ent, eps_high, agg, agg_norm, group_size, ...); logp_old and
    ref_logp are per-token [B*T] tensors.

    Returns dict(loss: float64[1] device tensor, stats: float64[5] device
    tensor (loss, pg, kl, entropy, clip-fraction shares summed), n_tokens,
    logp, entropy: float32[B*T], dhidden: like hidden, dweight: float32 [V, D],
    seqs_per_chunk)."""
    R, D = hidden.shape
    V = weight.shape[0]
    assert R == B * T and weight.shape[1] == D
    dev = hidden.device
    group = int(loss_kw.get("group_size") or 1)
    S = seqs_per_chunk or _seqs_per_chunk(B, T, V, hidden.element_size(), group, chunk_bytes)
    if B % group or S % group:
        raise ValueError("chunks must hold whole groups of sequences")
    per_token_adv = adv.numel() == R and R != B
    counts = torch_api.count_tokens(mask, B, T)  # (N, B') of the whole batch, on the device
    logits = torch.empty((S * T, V), dtype=hidden.dtype, device=dev)
    dhidden = torch.empty_like(hidden)
    dweight = torch.zeros((V, D), dtype=torch.float32, device=dev)
    logp = torch.empty(R, dtype=torch.float32, device=dev)
    ent = torch.empty(R, dtype=torch.float32, device=dev)
    stats_sum = torch.zeros(5, dtype=torch.float64, device=dev)
    ws = torch_api.new_workspace(S * T, dev)
    st = torch_api.new_stats(dev)
    kw = dict(loss_kw)
    lo_all, rf_all = kw.pop("logp_old", None), kw.pop("ref_logp", None)
    for b0 in range(0, B, S):
        b1 = min(B, b0 + S)
        r0, r1 = b0 * T, b1 * T
        lg = logits[: r1 - r0]
        torch.matmul(hidden[r0:r1], weight.t(), out=lg)
        a = adv[r0:r1] if per_token_adv else adv[b0:b1]
        torch_api.policy_loss(lg, ids[r0:r1], mask[r0:r1], a, b1 - b0, T, V=V,
                              logp_old=lo_all[r0:r1] if lo_all is not None else None,
                              ref_logp=rf_all[r0:r1] if rf_all is not None else None,
                              dlogits=lg, logp_out=logp[r0:r1], entropy_out=ent[r0:r1],
                              workspace=ws, stats=st, global_counts=counts, **kw)
        stats_sum += st[:40].view(torch.float64)
        torch.matmul(lg, weight, out=dhidden[r0:r1])
        _accumulate_f32(dweight, lg.t(), hidden[r0:r1])
    return dict(loss=stats_sum[:1].clone(), stats=stats_sum, n_tokens=counts[0:1],
                logp=logp, entropy=ent, dhidden=dhidden, dweight=dweight, seqs_per_chunk=S)


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
