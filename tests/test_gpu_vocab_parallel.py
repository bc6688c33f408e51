"""Vocabulary parallelism: the logits columns split into shards, each shard
launched twice (its partial row statistics, then, with every shard's
partials gathered in order, the loss and its own gradient columns).  Run
here as consecutive launches on one GPU, the shards together must give what
the oracle computes on the whole vocabulary: loss and statistics, logp and
entropy on every row, and every gradient element."""
import numpy as np
import pytest
import torch

import oracle
import ppo_policy_loss_gb300 as rl
from ppo_policy_loss_gb300 import synth, torch_api
from _parity import *  # noqa: F401,F403

pytestmark = pytest.mark.gpu

W = synth.WORKLOADS


@pytest.fixture(scope="module", autouse=True)
def _built():
    rl.build()
    rl.load()


CASES = {
    # streamed rows, three uneven shards (offsets multiples of 8 elements)
    "bf16_qwen_3shards": (W["qwen3_0p6b_grpo"].scaled(n_prompts=2, group=4, T=8,
                                                      lengths=("uniform", 2, 8), c_ent=0.01),
                          [0, 50000, 100008, 151936]),
    # resident rows (each shard of 16000 fp16 logits fits on chip), group rewards
    "f16_32000_2shards": (W["long_seq_grpo"].scaled(T=16, lengths=("uniform", 1, 16), beta=0.05),
                          [0, 16000, 32000]),
    # fp32, per-token advantages, a shard with a ragged tail
    "f32_ppo_2shards": (W["ppo_gae"].scaled(dtype="f32", V=5000, n_prompts=4, T=8),
                        [0, 2504, 5000]),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_vocab_shards_match_the_whole_vocabulary(name):
    w, cuts = CASES[name]
    small, logits = build_case(w)
    V, R, B, T = w.V, w.R, w.B, w.T
    mask, ids = small["mask"], small["ids"]
    arow, adv = adv_rows(w, small)
    host = storage_np(logits)[:, :V]
    lse, logp, ent = oracle.row_stats(host, w.dtype, V, ids, mask)
    lo, rf = composed_old_ref(logp, small, mask, R)
    rf_arg = rf if w.beta != 0 else None
    ref = oracle.loss_from_stats(logp, ent, mask, arow, lo, rf_arg, w.eps, w.beta, w.c_ent)
    band = band_mask(ref, w.eps) & (mask != 0)
    N = ref["n_tokens"]

    group_rewards = name.startswith("f16")
    a = to_dev(small["rewards"]) if group_rewards else to_dev(adv.astype(np.float32).reshape(-1))
    opts = dict(logp_old=to_dev(lo), ref_logp=to_dev(rf) if rf_arg is not None else None,
                eps=w.eps, beta=w.beta, c_ent=w.c_ent, grad_scale=float(N))
    if group_rewards:
        opts["group_size"] = w.group
    d_ids, d_mask = to_dev(ids), to_dev(mask)
    n = len(cuts) - 1
    parts = torch.empty((n, R, 4), dtype=torch.float32, device="cuda")
    for k in range(n):
        torch_api.policy_loss(logits[:, cuts[k]:cuts[k + 1]], d_ids, d_mask, a, B, T,
                              vocab_offset=cuts[k], vocab_total=V, partials_out=parts[k], **opts)
    dl = torch.full_like(logits, 7.0)
    outs = []
    for k in range(n):
        outs.append(torch_api.policy_loss(logits[:, cuts[k]:cuts[k + 1]], d_ids, d_mask, a, B, T,
                                          vocab_offset=cuts[k], vocab_total=V,
                                          shard_partials=parts,
                                          dlogits=dl[:, cuts[k]:cuts[k + 1]], **opts))
    torch.cuda.synchronize()
    for o in outs:  # every shard reports the whole loss
        assert_stats_match(torch_api.read_stats(o["stats"]), ref, int(band.sum()))
        assert_rows_close(o["logp"].cpu().numpy(), o["entropy"].cpu().numpy(), ref, mask)
    rows = np.arange(R)  # every row; a clip-band row may match either branch (all shards alike)
    scale = np.where(mask != 0, 1.0, 0.0)
    check_dlogits_rows(dl[:, :V], host, w.dtype, V, ids, rows, lse, ent, ref_rows(ref, rows), band,
                       scale, w.c_ent, where=name)


def test_vocab_shard_argument_errors():
    w = W["tiny_grpo"]
    small, logits = build_case(w)
    t = lambda x: to_dev(x)
    part = torch.empty((w.R, 4), dtype=torch.float32, device="cuda")
    with pytest.raises(rl.RlLossError):  # the shard runs past the vocabulary
        torch_api.policy_loss(logits, t(small["ids"]), t(small["mask"]), t(small["rewards"]),
                              w.B, w.T, vocab_offset=8, vocab_total=w.V, partials_out=part)
    with pytest.raises(rl.RlLossError):  # both launches at once
        torch_api.policy_loss(logits, t(small["ids"]), t(small["mask"]), t(small["rewards"]),
                              w.B, w.T, partials_out=part, shard_partials=part[None])
