"""GPU parity: the CUDA path (through the C ABI) against the fp64 CPU oracle.

Small cases compare every output element by element (loss and statistics,
per-token logp and entropy, every dlogits element at grad_scale 1 and N);
they are sized to span several 16 KB chunks, both row layouts (rows held
on chip for both passes, and rows streamed twice through the ring, up to
256 chunks per row), ragged vocabulary tails and padded rows.  The
full-size workloads run in the launch configuration the benchmark times and
are compared on the scalar loss and statistics (all rows), on logp/entropy
(all rows), on sampled dlogits rows, and on properties that hold at any size
(masked rows exactly zero).
"""
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


def _run_both(w, ld=None, grad_scales=(1.0, "N"), in_place=False, with_old=True,
              with_ref=None):
    """Full element-wise parity for a small workload."""
    small, logits = build_case(w, ld=ld)
    V, R, B, T = w.V, w.R, w.B, w.T
    ldv = logits.stride(0)
    mask, ids = small["mask"], small["ids"]
    arow, adv = adv_rows(w, small)
    host = storage_np(logits)[:, :V]
    lse, logp, ent = oracle.row_stats(host, w.dtype, V, ids, mask)
    lo, rf = composed_old_ref(logp, small, mask, R)
    with_ref = (w.beta != 0) if with_ref is None else with_ref
    lo_arg = lo if with_old else None
    rf_arg = rf if with_ref else None
    ref = oracle.loss_from_stats(logp, ent, mask, arow, lo_arg, rf_arg, w.eps, w.beta, w.c_ent)
    band = band_mask(ref, w.eps) & (mask != 0)
    n_band = int(band.sum())

    d_ids, d_mask = to_dev(ids), to_dev(mask)
    d_adv = to_dev(adv.astype(np.float32).reshape(-1))
    d_lo = to_dev(lo) if with_old else None
    d_rf = to_dev(rf) if with_ref else None
    N = ref["n_tokens"]
    report = {}
    for gs in grad_scales:
        gsv = float(N if gs == "N" else gs)
        src = logits.clone() if in_place else logits
        dst = src if in_place else torch.full_like(logits, 7.0)  # sentinel in padding columns
        out = torch_api.policy_loss(src, d_ids, d_mask, d_adv, B, T, V=V, logp_old=d_lo,
                                    ref_logp=d_rf, eps=w.eps, beta=w.beta, c_ent=w.c_ent,
                                    grad_scale=gsv, dlogits=dst)
        torch.cuda.synchronize()
        st = torch_api.read_stats(out["stats"])
        assert_stats_match(st, ref, n_band)
        assert_rows_close(out["logp"].cpu().numpy(), out["entropy"].cpu().numpy(), ref, mask)
        keep = ~band  # rows whose clip decision may flip are compared separately
        rows = np.nonzero(keep)[0]
        scale = np.where(mask[rows] != 0, gsv / N if N else 0.0, 0.0)
        d_ref = oracle.dlogits_rows(host, w.dtype, V, ids, rows, lse[rows], ent[rows],
                                    ref["g"][rows], scale, w.c_ent, w.dtype)
        d_gpu = storage_np(out["dlogits"][:, :V])[rows]
        report[gs] = assert_dlogits_close(d_gpu, d_ref, w.dtype, where=f"{w.name} gs={gs}")
        assert np.all(storage_np(out["dlogits"][:, :V])[mask == 0] == 0)
        if ldv != V and not in_place:  # padding columns are never written
            assert bool((out["dlogits"][:, V:] == 7.0).all())
    return report


SMALL = {
    "tiny_grpo_f32": W["tiny_grpo"],
    "qwen_vocab_bf16_c2": W["qwen3_0p6b_grpo"].scaled(n_prompts=2, group=4, T=8,
                                                      lengths=("uniform", 2, 8), c_ent=0.01),
    "qwen_vocab_f32_c4": W["tiny_grpo"].scaled(V=151936, T=4, lengths=("uniform", 1, 4)),
    "bf16_v200000_c3": W["large_grpo"].scaled(V=200000, n_prompts=1, group=8, T=4,
                                              lengths=("uniform", 1, 4), c_ent=0.02),
    "f16_v32000_c1": W["long_seq_grpo"].scaled(T=32, lengths=("geometric", 20, 32)),
    "ppo_gae_bf16": W["ppo_gae"].scaled(n_prompts=6, T=8),
    "f32_v12345_ragged": W["tiny_grpo"].scaled(V=12345),
    "bf16_v1001_ragged": W["qwen3_0p6b_grpo"].scaled(n_prompts=2, group=2, T=16, V=1001,
                                                     lengths=("uniform", 0, 16), c_ent=0.05),
    "f16_v7_tiny": W["long_seq_grpo"].scaled(n_prompts=2, group=4, T=8, V=7,
                                             lengths=("uniform", 1, 8), beta=0.1),
    "bf16_single_chunk": W["qwen3_0p6b_grpo"].scaled(n_prompts=2, group=4, T=8, V=8192,
                                                     lengths=("uniform", 1, 8)),
    "f32_v1M_stream": W["tiny_grpo"].scaled(n_prompts=1, group=2, T=4, V=1 << 20,
                                            lengths=("uniform", 1, 4)),
    "bf16_v300001_stream": W["large_grpo"].scaled(n_prompts=1, group=4, T=4, V=300001,
                                                  lengths=("uniform", 1, 4), c_ent=0.01),
    "f16_v49152_resident": W["long_seq_grpo"].scaled(n_prompts=1, group=4, T=8, V=49152,
                                                     lengths=("uniform", 2, 8)),
}
PADDED_LD = {"f32_v12345_ragged": 12348, "bf16_v1001_ragged": 1008, "f16_v7_tiny": 8,
             "bf16_v300001_stream": 300008}


@pytest.mark.parametrize("name", sorted(SMALL))
def test_small_parity(name):
    w = SMALL[name]
    _run_both(w, ld=PADDED_LD.get(name))


def test_launch_shape():
    # rows that fit the ring twice stay on chip in one CTA; longer rows are
    # streamed by one CTA; the persistent grid fills the device
    for dt, V in (("bf16", 151936), ("f32", 151936), ("bf16", 200000), ("f16", 32000),
                  ("f32", 1024), ("f32", 1 << 20)):
        c, n, smem = rl.rl_policy_loss_launch_shape(dt, V, 32768)
        assert c == 1 and 1 <= n <= 2048 and smem <= 227 * 1024, (dt, V, c, n, smem)
    assert rl.rl_policy_loss_launch_shape("bf16", 151936, 5)[1] == 5  # no more CTAs than rows
    with pytest.raises(rl.RlLossError):
        rl.rl_policy_loss_launch_shape("bf16", (1 << 30) + 8, 10)  # beyond 32-bit row offsets


def test_in_place_matches():
    _run_both(SMALL["qwen_vocab_bf16_c2"], grad_scales=("N",), in_place=True)


def test_on_policy_and_no_reference():
    _run_both(SMALL["bf16_v200000_c3"].scaled(beta=0.0), grad_scales=("N",), with_old=False,
              with_ref=False)


def test_deterministic_bitwise():
    w = SMALL["qwen_vocab_bf16_c2"]
    small, logits = build_case(w)
    args = (to_dev(small["ids"]), to_dev(small["mask"]),
            to_dev(oracle.group_advantages(small["rewards"], w.group).astype(np.float32)))
    outs = []
    for _ in range(2):
        o = torch_api.policy_loss(logits, *args, w.B, w.T, eps=w.eps, c_ent=0.01, grad_scale=7.0)
        torch.cuda.synchronize()
        outs.append((o["dlogits"].view(torch.int16).cpu(), o["stats"].cpu(), o["logp"].cpu()))
    for a, b in zip(*outs):
        assert torch.equal(a, b)


def test_forward_only_and_zero_valid_tokens_and_empty_batch():
    w = SMALL["bf16_v1001_ragged"]
    small, logits = build_case(w, ld=1008)
    ids, adv = to_dev(small["ids"]), to_dev(np.ones(w.B, np.float32))
    # forward only: no dlogits, same loss as with dlogits
    m = to_dev(small["mask"])
    a = torch_api.policy_loss(logits, ids, m, adv, w.B, w.T, V=w.V, c_ent=0.05, dlogits=None)
    b = torch_api.policy_loss(logits, ids, m, adv, w.B, w.T, V=w.V, c_ent=0.05)
    sa, sb = torch_api.read_stats(a["stats"]), torch_api.read_stats(b["stats"])
    assert sa == sb
    # N = 0: loss 0, every gradient element 0
    z = torch.zeros_like(m)
    o = torch_api.policy_loss(logits, ids, z, adv, w.B, w.T, V=w.V, c_ent=0.05, beta=0.1,
                              ref_logp=torch.zeros(w.R, device="cuda"))
    st = torch_api.read_stats(o["stats"])
    assert st["loss"] == 0 and st["n_tokens"] == 0 and st["device_error"] == 0
    assert int(torch.count_nonzero(o["dlogits"][:, :w.V])) == 0
    # B = 0: nothing to do, stats written
    e = torch.empty(0, 1008, dtype=logits.dtype, device="cuda")
    o = torch_api.policy_loss(e, ids[:0], m[:0], adv[:0], 0, w.T, V=w.V)
    st = torch_api.read_stats(o["stats"])
    assert st["n_tokens"] == 0 and st["loss"] == 0


def test_id_out_of_range_is_reported_not_trapped():
    w = SMALL["bf16_single_chunk"]
    small, logits = build_case(w)
    ids = small["ids"].copy()
    mask = small["mask"].copy()
    bad = int(np.nonzero(mask)[0][0])
    ids[bad] = w.V + 5
    masked = np.nonzero(mask == 0)[0]
    if masked.size:
        ids[masked[0]] = -7  # ignored: masked rows never read their id
    o = torch_api.policy_loss(logits, to_dev(ids), to_dev(mask),
                              to_dev(np.ones(w.B, np.float32)), w.B, w.T)
    st = torch_api.read_stats(o["stats"])
    assert st["device_error"] == rl.RL_DEVERR_ID_RANGE
    assert rl.rl_read_device_status(o["workspace"]) == rl.RL_ERR_ID_RANGE
    lp = o["logp"].cpu().numpy()
    assert np.isnan(lp[bad]) and np.isnan(st["loss"])
    assert torch.isnan(o["dlogits"][bad].float()).all()
    others = np.nonzero(mask)[0][1:]
    assert np.isfinite(lp[others]).all()
    # the next call on the same workspace starts clean
    ids[bad] = 0
    o2 = torch_api.policy_loss(logits, to_dev(ids), to_dev(mask), to_dev(np.ones(w.B, np.float32)),
                               w.B, w.T, workspace=o["workspace"])
    assert torch_api.read_stats(o2["stats"])["device_error"] == 0
    assert rl.rl_read_device_status(o2["workspace"]) == rl.RL_OK


# ----------------------------------------------------------------- advantages
@pytest.mark.parametrize("name", sorted(n for n in W if W[n].advantage == "group"))
def test_group_advantages_workloads(name):
    w = W[name]
    small = synth.small_inputs(w)
    ref = oracle.group_advantages(small["rewards"], w.group)
    got = torch_api.group_advantages(to_dev(small["rewards"]), w.group).cpu().numpy()
    assert np.all(np.abs(got - ref) <= ADV_TOL * np.maximum(np.abs(ref), 1.0))
    assert np.all(got[ref == 0] == 0)


@pytest.mark.parametrize("G,ddof", [(1, 0), (2, 1), (5, 1), (33, 1), (300, 0), (1000, 1)])
def test_group_advantages_shapes(G, ddof):
    rng = np.random.default_rng(G)
    R = rng.random(7 * G).astype(np.float32)
    R[:G] = 0.5  # one group of equal rewards -> exactly zero
    ref = oracle.group_advantages(R, G, 1e-4, ddof)
    d = to_dev(R)
    got = torch_api.group_advantages(d, G, ddof=ddof).cpu().numpy()
    assert np.all(np.abs(got - ref) <= ADV_TOL * np.maximum(np.abs(ref), 1.0))
    assert np.all(got[:G] == 0)
    torch_api.group_advantages(d, G, ddof=ddof, out=d)  # in place
    assert np.array_equal(d.cpu().numpy(), got)


@pytest.mark.parametrize("T,gamma,lam", [(512, 1.0, 0.95), (37, 0.99, 0.9), (1000, 1.0, 1.0),
                                         (5, 0.5, 0.0), (1, 1.0, 0.95)])
def test_gae_parity(T, gamma, lam):
    rng = np.random.default_rng(T)
    B = 70
    r = rng.normal(0, 1, (B, T)).astype(np.float32)
    v = rng.normal(0, 0.5, (B, T)).astype(np.float32)
    L = rng.integers(0, T + 1, B).astype(np.int32)
    L[0], L[1] = T, 0
    L[2] = T + 9  # clamped to T
    A, ret = oracle.gae(r, v, L, float(np.float32(gamma)), float(np.float32(lam)))
    a, rt = torch_api.gae(to_dev(r), to_dev(v), to_dev(L), gamma, lam)
    a, rt = a.cpu().numpy(), rt.cpu().numpy()
    assert np.all(np.abs(a - A) <= ADV_TOL * np.maximum(np.abs(A), 1.0))
    assert np.all(np.abs(rt - ret) <= ADV_TOL * np.maximum(np.abs(ret), 1.0))


def test_gae_ppo_workload():
    w = W["ppo_gae"]
    small = synth.small_inputs(w)
    A, ret = oracle.gae(small["rewards"], small["values"], small["lengths"], w.gamma, w.lam)
    a, rt = torch_api.gae(to_dev(small["rewards"]), to_dev(small["values"]),
                          to_dev(small["lengths"]), w.gamma, w.lam)
    assert np.all(np.abs(a.cpu().numpy() - A) <= ADV_TOL * np.maximum(np.abs(A), 1.0))
    assert np.all(np.abs(rt.cpu().numpy() - ret) <= ADV_TOL * np.maximum(np.abs(ret), 1.0))
    a2, r2 = torch_api.gae(to_dev(small["rewards"]), to_dev(small["values"]),
                           to_dev(small["lengths"]), w.gamma, w.lam, want_returns=False)
    assert r2 is None and torch.equal(a2, a)


# ----------------------------------------------------------------- full size
FULL = ["qwen3_0p6b_grpo", "long_seq_grpo", "ppo_gae", "large_grpo"]


@pytest.mark.parametrize("name", FULL)
def test_full_size_workload(name):
    """The benchmark's launch configuration at the workload's full size."""
    w = W[name]
    small = synth.small_inputs(w)
    logits = synth.logits(w, device="cuda")
    V, R = w.V, w.R
    mask, ids = small["mask"], small["ids"]
    arow, adv = adv_rows(w, small)
    lse, logp, ent = oracle_stats_chunked(logits, w.dtype, V, ids, mask)
    lo, rf = composed_old_ref(logp, small, mask, R)
    rf_arg = rf if w.beta != 0 else None
    ref = oracle.loss_from_stats(logp, ent, mask, arow, lo, rf_arg, w.eps, w.beta, w.c_ent)
    band = band_mask(ref, w.eps) & (mask != 0)
    N = ref["n_tokens"]
    if w.advantage == "gae":  # the GPU computes the advantages it consumes
        d_adv, _ = torch_api.gae(to_dev(small["rewards"]), to_dev(small["values"]),
                                 to_dev(small["lengths"]), w.gamma, w.lam, want_returns=False)
        assert np.all(np.abs(d_adv.cpu().numpy() - adv) <= ADV_TOL * np.maximum(np.abs(adv), 1.0))
        d_adv = d_adv.reshape(-1)
    else:
        d_adv = torch_api.group_advantages(to_dev(small["rewards"]), w.group)
    out = torch_api.policy_loss(logits, to_dev(ids), to_dev(mask), d_adv, w.B, w.T,
                                logp_old=to_dev(lo), ref_logp=to_dev(rf) if rf_arg is not None else None,
                                eps=w.eps, beta=w.beta, c_ent=w.c_ent, grad_scale=float(N))
    torch.cuda.synchronize()
    st = torch_api.read_stats(out["stats"])
    assert_stats_match(st, ref, int(band.sum()))
    assert_rows_close(out["logp"].cpu().numpy(), out["entropy"].cpu().numpy(), ref, mask)
    rows = np.array([r for r in valid_and_masked_sample(mask, 24, seed=w.seed) if not band[r]])
    host = storage_np(logits.index_select(0, to_dev(rows)))
    scale = np.where(mask[rows] != 0, 1.0, 0.0)
    d_ref = oracle.dlogits_rows(host, w.dtype, V, ids[rows], np.arange(rows.size), lse[rows],
                                ent[rows], ref["g"][rows], scale, w.c_ent, w.dtype)
    d_gpu = storage_np(out["dlogits"].index_select(0, to_dev(rows)))
    assert_dlogits_close(d_gpu, d_ref, w.dtype, where=name)
    # every masked row is exactly zero (checked on the device, in chunks)
    dm = to_dev(mask == 0)
    for r0 in range(0, R, 4096):
        blk = out["dlogits"][r0:r0 + 4096][dm[r0:r0 + 4096]]
        assert int(torch.count_nonzero(blk.view(torch.int16))) == 0
