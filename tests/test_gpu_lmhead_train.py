"""The policy loss from hidden states in chunks of sequences
(ppo_policy_loss_gb300.lmhead_train): library GEMMs for the logits and the
two gradient products, the fused loss kernel in place in between.  The
oracle gets the very logits the GEMM produced (the same GEMM call per chunk
gives the same bits), so the loss, log-probs and entropies are held to the
usual tolerances; the hidden-state and weight gradients are compared with
the fp64 products of the oracle's dlogits, within bf16 GEMM rounding."""
import numpy as np
import pytest
import torch

import oracle
import ppo_policy_loss_gb300 as rl
from ppo_policy_loss_gb300 import lmhead_train, synth
from _parity import LOGP_ATOL, assert_scalar_close, storage_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    rl.build()
    rl.load()


@pytest.mark.parametrize("agg,group_rewards", [("token_mean", False), ("seq_mean_token_mean", True)])
def test_lmhead_policy_loss_chunks_match_the_oracle(agg, group_rewards):
    dev = torch.device("cuda:0")
    w = synth.WORKLOADS["qwen3_0p6b_grpo"].scaled(n_prompts=2, group=4, T=64, V=20000,
                                                   lengths=("uniform", 8, 64), c_ent=0.01,
                                                   seed=321)
    B, T, V, R, D = w.B, w.T, w.V, w.R, 256
    small = synth.small_inputs(w)
    hidden, weight, _ = synth.lmhead_inputs(R, D, V, 322, 3.0)
    ids, mask = small["ids"], small["mask"]
    h, W_ = hidden.to(dev), weight.to(dev)
    S = 4  # two chunks of one group each
    # the logits each chunk's GEMM produces
    lg = torch.cat([torch.matmul(h[b0 * T:(b0 + S) * T], W_.t()) for b0 in range(0, B, S)])
    host = storage_np(lg)
    lse, logp, ent = oracle.row_stats(host, "bf16", V, ids, mask)
    A = oracle.group_advantages(small["rewards"], w.group)
    lo = np.where(mask != 0, logp + small["noise_old"], 0.0).astype(np.float32)
    rf = np.where(mask != 0, logp + small["noise_ref"], 0.0).astype(np.float32)
    ref = oracle.loss_from_stats(logp, ent, mask, np.repeat(A, T), lo, rf, w.eps, w.beta,
                                 w.c_ent, agg=agg, T=T)
    t = lambda x: torch.from_numpy(np.ascontiguousarray(x)).to(dev)
    adv = t(small["rewards"]) if group_rewards else t(A.astype(np.float32))
    opts = dict(logp_old=t(lo), ref_logp=t(rf), eps=w.eps, beta=w.beta, c_ent=w.c_ent, agg=agg,
                grad_scale=1.0)
    if group_rewards:
        opts["group_size"] = w.group
    out = lmhead_train.lmhead_policy_loss(h, W_, t(ids), t(mask), adv, B, T, seqs_per_chunk=S,
                                          **opts)
    torch.cuda.synchronize()
    assert out["seqs_per_chunk"] == S
    assert_scalar_close("loss", float(out["loss"][0]), ref["loss"])
    mb = mask != 0
    assert np.abs(out["logp"].cpu().numpy()[mb] - logp[mb]).max() <= LOGP_ATOL
    assert np.abs(out["entropy"].cpu().numpy()[mb] - ent[mb]).max() <= LOGP_ATOL
    # gradients: dlogits from the oracle (fp64), then the exact products
    scale = ref["weights"] * mask  # grad_scale 1: the loss weight of each token
    d_ref = oracle.dlogits_rows(host, "bf16", V, ids, np.arange(R), lse, ent, ref["g"], scale,
                                w.c_ent, "f64")
    Wd = oracle.decode(storage_np(weight), "bf16")
    Hd = oracle.decode(storage_np(hidden), "bf16")
    dh_ref, dw_ref = d_ref @ Wd, d_ref.T @ Hd
    dh = oracle.decode(storage_np(out["dhidden"]), "bf16")
    dw = out["dweight"].cpu().numpy().astype(np.float64)
    for name, got, exp in (("dhidden", dh, dh_ref), ("dweight", dw, dw_ref)):
        rel = np.linalg.norm(got - exp) / np.linalg.norm(exp)
        assert rel <= 1e-2, (name, rel)
        assert np.abs(got - exp).max() <= 3e-2 * np.abs(exp).max(), name

    # the autograd wrapper hands back the same gradients
    hv = h.clone().requires_grad_(True)
    Wv = W_.clone().requires_grad_(True)
    loss = lmhead_train.LMHeadPolicyLoss.apply(hv, Wv, t(ids), t(mask), adv, B, T,
                                               dict(opts, seqs_per_chunk=S))
    loss.backward()
    assert torch.equal(hv.grad, out["dhidden"])
    assert torch.equal(Wv.grad, out["dweight"].to(Wv.dtype))


def test_lmhead_policy_loss_default_chunks():
    """Without an explicit chunk the op picks whole groups within chunk_bytes and
    the result does not depend on the chunking beyond GEMM rounding (the
    library may round a 64-row and a 256-row product's bf16 logits
    differently: up to half an ulp of |z| ~ 3, so 1e-2 bounds logp here)."""
    dev = torch.device("cuda:0")
    B, T, V, D = 8, 32, 8000, 128
    R = B * T
    hidden, weight, ids = synth.lmhead_inputs(R, D, V, 5, 2.0)
    h, W_, i = hidden.to(dev), weight.to(dev), ids.to(dev)
    mask = torch.ones(R, dtype=torch.uint8, device=dev)
    adv = torch.linspace(-1, 1, B, device=dev)
    a = lmhead_train.lmhead_policy_loss(h, W_, i, mask, adv, B, T, chunk_bytes=2 * T * V * 2)
    b = lmhead_train.lmhead_policy_loss(h, W_, i, mask, adv, B, T, chunk_bytes=1 << 30)
    assert a["seqs_per_chunk"] == 2 and b["seqs_per_chunk"] == B
    torch.cuda.synchronize()
    la, lb = float(a["loss"][0]), float(b["loss"][0])
    assert abs(la - lb) <= 1e-2 * max(1e-3, abs(lb)), (la, lb)
    assert torch.allclose(a["logp"], b["logp"], atol=1e-2)
    assert torch.allclose(a["dhidden"].float(), b["dhidden"].float(), atol=1e-2 * float(b["dhidden"].abs().max()))
