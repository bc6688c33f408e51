"""The policy loss through the LM head on the tensor cores: the three backward
GEMMs (rl_lmhead_dlogits, rl_lmhead_dhidden, rl_lmhead_dweight), the row
statistics (rl_lmhead_row_partials) and the training op built on them
(ppo_policy_loss_gb300.lmhead_train), against the fp64 oracle.

GEMM outputs are compared element by element with a bound derived from fp32
accumulation of exact 16-bit products (_parity.accumulation_bound) plus the
output's own rounding; the gradient dz with the dlogits tolerance (1 ulp +
1e-6) of the loss kernel; the chain's dhidden and dweight with the bound
propagated from dz's rounding through the product."""
import numpy as np
import pytest
import torch

import oracle
import ppo_policy_loss_gb300 as rl
from ppo_policy_loss_gb300 import lmhead_train, synth, torch_api
from _parity import (LOGP_ATOL, DLOGIT_ATOL, accumulation_bound, assert_scalar_close,
                     rows_within, storage_np, to_dev)

pytestmark = pytest.mark.gpu

DT = {"bf16": torch.bfloat16, "f16": torch.float16}


@pytest.fixture(scope="module", autouse=True)
def _built():
    rl.build()
    rl.load()


def _rand16(shape, sd, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(shape, generator=g) * sd).to(DT[dtype])


def _dec(t, dtype):
    return oracle.decode(storage_np(t), dtype)


def _assert_within(got, exp, tol, where):
    err = np.abs(got - exp)
    bad = ~(err <= tol)
    if bad.any():
        i = tuple(np.argwhere(bad)[0])
        raise AssertionError(f"{where}: {int(bad.sum())} of {bad.size} out of bound; first {i}: "
                             f"got {got[i]!r} exact {exp[i]!r} bound {tol[i]!r}")
    return float((err / np.maximum(tol, 1e-300)).max())


# ----------------------------------------------------------------- the two products
def _padded(t, ld):
    """A device copy of t [rows, n] in rows of ld >= n elements (padding 7.0)."""
    out = torch.full((t.shape[0], ld), 7.0, dtype=t.dtype, device="cuda")
    out[:, :t.shape[1]] = t.cuda()
    return out


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("R,D,V", [(512, 256, 20000), (300, 200, 1000), (129, 8, 77)])
def test_dhidden_is_the_product_within_fp32_accumulation(dtype, R, D, V):
    """dH = dz @ W with M, N and K tails (K = V); dz rows padded to a multiple of 8."""
    dz = _rand16((R, V), 0.05, dtype, R + V)
    W = _rand16((V, D), 0.1, dtype, D + 1)
    ld_dz = -(-V // 8) * 8
    dH = torch.full((R, D), 7.0, dtype=DT[dtype], device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    rl.rl_lmhead_dhidden(_padded(dz, ld_dz), ld_dz, W.cuda(), D, dtype, R, D, V, dH, D, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    A, B = _dec(dz, dtype), _dec(W, dtype)
    exact = A @ B
    tol = oracle.ulp(exact, dtype) + accumulation_bound(A, B)
    _assert_within(_dec(dH, dtype), exact, tol, f"dhidden {dtype} {R}x{D}x{V}")


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("R,D,V", [(512, 256, 20000), (300, 200, 1000), (77, 8, 129)])
def test_dweight_is_the_product_within_fp32_accumulation(dtype, R, D, V):
    """dW = dz^T @ hidden written, then a second chunk's product added to it
    (M = V, N = D, K = R, with tails)."""
    dz1, dz2 = _rand16((R, V), 0.05, dtype, 3 * R), _rand16((R, V), 0.05, dtype, 3 * R + 1)
    h1, h2 = _rand16((R, D), 1.0, dtype, 5 * D), _rand16((R, D), 1.0, dtype, 5 * D + 1)
    ld_dz = -(-V // 8) * 8  # dz rows padded to a multiple of 8 elements
    dW = torch.full((V, D), 7.0, dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    rl.rl_lmhead_dweight(_padded(dz1, ld_dz), ld_dz, h1.cuda(), D, dtype, R, D, V, dW, D, False,
                         status)
    torch.cuda.synchronize()
    A1, B1 = _dec(dz1, dtype).T, _dec(h1, dtype)
    first = A1 @ B1
    b1 = accumulation_bound(A1, B1)
    _assert_within(dW.cpu().numpy().astype(np.float64), first, b1, f"dweight {dtype} write")
    rl.rl_lmhead_dweight(_padded(dz2, ld_dz), ld_dz, h2.cuda(), D, dtype, R, D, V, dW, D, True,
                         status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    A2, B2 = _dec(dz2, dtype).T, _dec(h2, dtype)
    both = first + A2 @ B2
    tol = b1 + accumulation_bound(A2, B2) + 2.0 ** -23 * np.abs(both)  # + the fp32 add of the chunks
    _assert_within(dW.cpu().numpy().astype(np.float64), both, tol, f"dweight {dtype} accumulate")


# ----------------------------------------------------------------- row statistics and dz
def _chain_case(seed=321, V=20000, D=256, dtype="bf16", T=64):
    w = synth.WORKLOADS["qwen3_0p6b_grpo"].scaled(n_prompts=2, group=4, T=T, V=V,
                                                   lengths=("uniform", 8, T), c_ent=0.01,
                                                   seed=seed)
    small = synth.small_inputs(w)
    hidden, weight, _ = synth.lmhead_inputs(w.R, D, V, seed + 1, 3.0)
    if dtype != "bf16":
        hidden, weight = hidden.float().to(DT[dtype]), weight.float().to(DT[dtype])
    return w, small, hidden, weight


def _oracle_chain(w, small, hidden, weight, dtype, grad_scale, agg="token_mean"):
    """The oracle's loss and gradients on its own fp64 logits; logp_old / ref
    from the oracle's logp plus the workload's noise."""
    z = oracle.lmhead_logits(storage_np(hidden), storage_np(weight), dtype)
    ids, mask = small["ids"], small["mask"]
    _, logp, _ = oracle.row_stats(z, "f64", w.V, ids, mask)
    lo = np.where(mask != 0, logp + small["noise_old"], 0.0).astype(np.float32)
    rf = np.where(mask != 0, logp + small["noise_ref"], 0.0).astype(np.float32)
    A = oracle.group_advantages(small["rewards"], w.group)
    ref = oracle.lmhead_policy_loss(storage_np(hidden), storage_np(weight), dtype, ids, mask,
                                    np.repeat(A, w.T), lo, rf, w.eps, w.beta, w.c_ent,
                                    grad_scale=grad_scale, agg=agg, T=w.T)
    return ref, lo, rf, A


def test_row_partials_give_the_oracle_row_statistics():
    w, small, hidden, weight = _chain_case()
    R, V, D = w.R, w.V, hidden.shape[1]
    parts = torch.empty((R, 4), dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = torch.zeros(max(16, rl.rl_lmhead_workspace_size(R, V)), dtype=torch.uint8, device="cuda")
    ids = small["ids"]
    rl.rl_lmhead_row_partials(hidden.cuda(), D, weight.cuda(), D, "bf16", R, D, V, to_dev(ids), parts,
                              status, ws, ws.numel())
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    m, S, Tt, zy = parts.cpu().numpy().astype(np.float64).T
    lse = m + np.log(S)
    H = np.log(2.0) * (np.log2(S) - Tt / S)
    r_lse, r_logp, r_H = oracle.lmhead_row_stats(storage_np(hidden), storage_np(weight), ids, "bf16")
    assert np.abs(lse - r_lse).max() <= LOGP_ATOL
    assert np.abs(zy - lse - r_logp).max() <= LOGP_ATOL
    assert np.abs(H - r_H).max() <= LOGP_ATOL


@pytest.mark.parametrize("dtype,T", [("bf16", 64), ("f16", 37)])
def test_dlogits_kernel_with_oracle_coefficients(dtype, T):
    """rl_lmhead_dlogits alone: the oracle's row coefficients in, every element
    of dz against the oracle's gradient rounded to the format (V = 3000: a
    partial last column tile; T = 37: 296 rows, a partial last row tile)."""
    w, small, hidden, weight = _chain_case(V=3000, D=128, dtype=dtype, seed=77, T=T)
    R, V, D = w.R, w.V, hidden.shape[1]
    N = int(small["mask"].sum())
    ref, lo, rf, A = _oracle_chain(w, small, hidden, weight, dtype, grad_scale=float(N))
    s = np.where(small["mask"] != 0, float(N) * ref["weights"], 0.0)
    ln2 = np.log(2.0)
    coef = np.stack([ref["lse"] / ln2, s * (ref["g"] + w.c_ent * ref["entropy"]), s * w.c_ent * ln2,
                     s * ref["g"]], axis=1).astype(np.float32)
    coef[small["mask"] == 0] = 0.0
    dz = torch.full((R, V), 7.0, dtype=DT[dtype], device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    rl.rl_lmhead_dlogits(hidden.cuda(), D, weight.cuda(), D, dtype, R, D, V, to_dev(small["ids"]),
                         to_dev(coef), dz, V, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    expect = oracle.encode(ref["dz"], dtype)
    ok, worst = rows_within(dz, expect, dtype)
    assert ok.all(), (int((~ok).sum()), worst)
    assert not bool((dz[torch.from_numpy(small["mask"] == 0).cuda()] != 0).any())


# ----------------------------------------------------------------- the training op
@pytest.mark.parametrize("agg,group_rewards", [("token_mean", False), ("seq_mean_token_mean", True)])
def test_lmhead_policy_loss_matches_the_oracle_chain(agg, group_rewards):
    w, small, hidden, weight = _chain_case()
    B, T, V, R, D = w.B, w.T, w.V, w.R, hidden.shape[1]
    ids, mask = small["ids"], small["mask"]
    N = int(mask.sum())
    gs = float(N)  # loss-scaled gradients: the ulp terms of the bounds bind
    ref, lo, rf, A = _oracle_chain(w, small, hidden, weight, "bf16", gs, agg)
    h, W_ = hidden.cuda(), weight.cuda()
    adv = to_dev(small["rewards"]) if group_rewards else to_dev(A.astype(np.float32))
    opts = dict(logp_old=to_dev(lo), ref_logp=to_dev(rf), eps=w.eps, beta=w.beta, c_ent=w.c_ent,
                agg=agg, grad_scale=gs)
    if group_rewards:
        opts["group_size"] = w.group
    out = lmhead_train.lmhead_policy_loss(h, W_, to_dev(ids), to_dev(mask), adv, B, T,
                                          seqs_per_chunk=3, **opts)
    torch.cuda.synchronize()
    assert int(out["status"].item()) == 0
    st = torch_api.read_stats(out["loss_stats"])
    assert st["device_error"] == 0 and st["n_tokens"] == N
    for k in ("loss", "pg_term", "kl_term", "ent_term"):
        assert_scalar_close(k, st[k], ref[k])
    mb = mask != 0
    assert np.abs(out["logp"].cpu().numpy()[mb] - ref["logp"][mb]).max() <= LOGP_ATOL
    assert np.abs(out["entropy"].cpu().numpy()[mb] - ref["entropy"][mb]).max() <= LOGP_ATOL
    assert np.all(out["logp"].cpu().numpy()[~mb] == 0)
    # dhidden and dweight: the GPU's dz is the oracle's within 1 ulp + 1e-6 per element
    # (the loss kernel's dlogits tolerance); that error, carried through the exact
    # product, plus fp32 accumulation and the output's rounding, bounds each element
    dz = ref["dz"]
    dz_err = oracle.ulp(dz, "bf16") + DLOGIT_ATOL
    Wd = oracle.decode(storage_np(weight), "bf16")
    Hd = oracle.decode(storage_np(hidden), "bf16")
    tol_h = (oracle.ulp(ref["dhidden"], "bf16") + dz_err @ np.abs(Wd) + accumulation_bound(dz, Wd))
    _assert_within(oracle.decode(storage_np(out["dhidden"]), "bf16"), ref["dhidden"], tol_h,
                   "chain dhidden")
    # dweight is accumulated in fp32 chunk by chunk (3 sequences each): each chunk's
    # product has its own accumulation bound, and adding it to the running total rounds once
    tol_w = dz_err.T @ np.abs(Hd)
    total = np.zeros_like(ref["dweight"])
    for r0 in range(0, R, 3 * T):
        sl = slice(r0, min(R, r0 + 3 * T))
        tol_w += accumulation_bound(dz[sl].T, Hd[sl])
        total += dz[sl].T @ Hd[sl]
        tol_w += 2.0 ** -23 * np.abs(total)
    _assert_within(out["dweight"].cpu().numpy().astype(np.float64), ref["dweight"], tol_w,
                   "chain dweight")

    # the autograd wrapper hands back the same gradients
    hv = h.clone().requires_grad_(True)
    Wv = W_.clone().requires_grad_(True)
    loss = lmhead_train.LMHeadPolicyLoss.apply(hv, Wv, to_dev(ids), to_dev(mask), adv, B, T,
                                               dict(opts, seqs_per_chunk=3))
    loss.backward()
    assert torch.equal(hv.grad, out["dhidden"])
    assert torch.equal(Wv.grad, out["dweight"].to(Wv.dtype))


def test_chunking_changes_only_the_weight_gradients_summation_order():
    """dz and dhidden are computed row by row: any chunking gives the same bits.
    dweight sums the chunks' products in another order: equal within fp32."""
    dev = torch.device("cuda:0")
    B, T, V, D = 8, 32, 8000, 128
    R = B * T
    hidden, weight, ids = synth.lmhead_inputs(R, D, V, 5, 2.0)
    h, W_, i = hidden.to(dev), weight.to(dev), ids.to(dev)
    mask = torch.ones(R, dtype=torch.uint8, device=dev)
    adv = torch.linspace(-1, 1, B, device=dev)
    a = lmhead_train.lmhead_policy_loss(h, W_, i, mask, adv, B, T, chunk_bytes=2 * T * V * 2)
    b = lmhead_train.lmhead_policy_loss(h, W_, i, mask, adv, B, T)
    torch.cuda.synchronize()
    assert a["seqs_per_chunk"] == 2 and b["seqs_per_chunk"] == B
    assert torch.equal(a["loss_stats"], b["loss_stats"])
    assert torch.equal(a["dhidden"], b["dhidden"])
    dw_a, dw_b = a["dweight"].double(), b["dweight"].double()
    assert float((dw_a - dw_b).abs().max()) <= 1e-5 * float(dw_b.abs().max())


def test_lmhead_policy_loss_qwen3_head_full_size_sampled_rows():
    """The training op at the Qwen3-0.6B head's full size (32 x 1024 rows, D 1024,
    V 151936 bf16) with the GRPO workload's mask, ids and rewards, in its default
    chunking.  The oracle recomputes 16 sampled valid rows one by one (their
    fp64 logits, statistics, gradient coefficients with the batch's token
    count and group advantages, dz and dhidden = dz W) and 4 masked rows; the
    loss and the counts hold over the whole batch."""
    dev = torch.device("cuda:0")
    w = synth.WORKLOADS["qwen3_0p6b_grpo"]
    B, T, V, R, D = w.B, w.T, w.V, w.R, 1024
    small = synth.small_inputs(w)
    ids, mask = small["ids"], small["mask"]
    hidden, weight, _ = synth.lmhead_inputs(R, D, V, 203, 3.0)
    Hs, Ws = storage_np(hidden), storage_np(weight)
    Wd = oracle.decode(Ws, "bf16")
    rng = np.random.default_rng(204)
    valid = np.nonzero(mask)[0]
    rows = np.unique(np.concatenate([rng.choice(valid, 14, replace=False), valid[[0, -1]]]))
    masked = rng.choice(np.nonzero(mask == 0)[0], 4, replace=False)
    # per sampled row: fp64 logits and statistics; logp_old / ref = that logp + the noise.
    # Other rows get seeded values far from their logp (inputs only: those rows are not compared).
    z = oracle.decode(Hs[rows], "bf16") @ Wd.T
    lse, logp, ent = oracle.row_stats(z, "f64", V, ids[rows], np.ones(rows.size, np.uint8))
    lo = np.where(mask != 0, -12.0 + small["noise_old"], 0.0)
    rf = np.where(mask != 0, -12.0 + small["noise_ref"], 0.0)
    lo[rows] = logp + small["noise_old"][rows]
    rf[rows] = logp + small["noise_ref"][rows]
    lo, rf = lo.astype(np.float32), rf.astype(np.float32)
    A = oracle.group_advantages(small["rewards"], w.group)
    N = int(mask.sum())
    out = lmhead_train.lmhead_policy_loss(hidden.to(dev), weight.to(dev), to_dev(ids), to_dev(mask),
                                          to_dev(small["rewards"]), B, T, logp_old=to_dev(lo),
                                          ref_logp=to_dev(rf), eps=w.eps, beta=w.beta,
                                          c_ent=0.01, group_size=w.group, grad_scale=float(N))
    torch.cuda.synchronize()
    assert int(out["status"].item()) == 0
    st = torch_api.read_stats(out["loss_stats"])
    assert st["device_error"] == 0 and st["n_tokens"] == N and np.isfinite(st["loss"])
    lp_gpu, h_gpu = out["logp"].cpu().numpy(), out["entropy"].cpu().numpy()
    assert np.abs(lp_gpu[rows] - logp).max() <= LOGP_ATOL
    assert np.abs(h_gpu[rows] - ent).max() <= LOGP_ATOL
    assert np.all(lp_gpu[mask == 0] == 0) and np.all(h_gpu[mask == 0] == 0)
    # the sampled rows' gradient coefficients, as the oracle's token objective gives them
    # (token_mean at grad_scale N: each valid row's scale is 1).  A row whose ratio lies
    # within the logp tolerance of a clip boundary may take either one-sided derivative.
    obj = oracle.token_objective(logp, ent, np.ones(rows.size, np.uint8), A[rows // T], lo[rows],
                                 rf[rows], w.eps, w.beta, 0.01)
    log_r = logp - lo[rows]
    band = np.zeros(rows.size, bool)
    for edge in (np.log1p(w.eps), np.log1p(-w.eps)):
        band |= np.abs(log_r - edge) <= LOGP_ATOL
    dh = oracle.decode(storage_np(out["dhidden"][torch.from_numpy(rows)]), "bf16")
    ok_any = np.zeros(rows.size, bool)
    variants = [obj["g"]] + ([obj["g_unclipped"], obj["g_clipped"]] if band.any() else [])
    for k, g in enumerate(variants):
        dz = oracle.dlogits_rows(z, "f64", V, ids[rows], np.arange(rows.size), lse, ent, g,
                                 np.ones(rows.size), 0.01, "f64")
        dh_ref = dz @ Wd
        dz_err = oracle.ulp(dz, "bf16") + DLOGIT_ATOL
        tol = oracle.ulp(dh_ref, "bf16") + dz_err @ np.abs(Wd) + accumulation_bound(dz, Wd)
        ok = (np.abs(dh - dh_ref) <= tol).all(axis=1)
        if k == 0:
            assert ok[~band].all(), _assert_within(dh[~band], dh_ref[~band], tol[~band],
                                                   "full-size dhidden")
        ok_any |= ok
    assert ok_any.all(), np.nonzero(~ok_any)[0]
    assert int(torch.count_nonzero(out["dhidden"][torch.from_numpy(masked)].view(torch.int16))) == 0
    assert bool(torch.isfinite(out["dweight"]).all())
