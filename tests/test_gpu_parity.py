"""GPU parity: the CUDA path (through the C ABI) against the fp64 CPU oracle.

Small cases compare every output element by element (loss and statistics,
per-token logp and entropy, every dlogits element at grad_scale 1 and N);
they are sized to span several 32 KB chunks, both row layouts (rows of at
most two chunks held on chip for both passes, longer rows streamed twice
through the ring, up to 128 chunks per row, including a row whose last
chunk is 16 bytes), ragged vocabulary tails and padded rows.  The
full-size workloads run in the launch configuration the benchmark times and
are compared on the scalar loss and statistics, on logp/entropy of every
row and on every element of every gradient row (masked rows exactly zero),
at grad_scale N and 1.  Rows whose ratio lies within CLIP_BAND of a clip
boundary must match the gradient of one of the surrogate's two branches.
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
              with_ref=None, ids=None):
    """Full element-wise parity for a small workload (``ids`` replaces the sampled ids)."""
    small, logits = build_case(w, ld=ld)
    if ids is not None:
        small["ids"] = np.asarray(ids, dtype=np.int64)
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
        rows = np.arange(R)  # every row; clip-band rows may match either branch
        scale = np.where(mask != 0, gsv / N if N else 0.0, 0.0)
        report[gs] = check_dlogits_rows(out["dlogits"][:, :V], host, w.dtype, V, ids, rows, lse,
                                        ent, ref_rows(ref, rows), band, scale, w.c_ent,
                                        where=f"{w.name} gs={gs}")
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
    "bf16_single_chunk": W["qwen3_0p6b_grpo"].scaled(n_prompts=2, group=4, T=8, V=16384,
                                                     lengths=("uniform", 1, 8)),
    "bf16_half_chunk": W["qwen3_0p6b_grpo"].scaled(n_prompts=2, group=4, T=8, V=8192,
                                                   lengths=("uniform", 1, 8)),
    "f32_v1M_stream": W["tiny_grpo"].scaled(n_prompts=1, group=2, T=4, V=1 << 20,
                                            lengths=("uniform", 1, 4)),
    "bf16_v300001_stream": W["large_grpo"].scaled(n_prompts=1, group=4, T=4, V=300001,
                                                  lengths=("uniform", 1, 4), c_ent=0.01),
    "f16_v32768": W["long_seq_grpo"].scaled(n_prompts=1, group=4, T=8, V=32768,
                                            lengths=("uniform", 2, 8)),
    "f16_v32776": W["long_seq_grpo"].scaled(n_prompts=1, group=4, T=8, V=32776,
                                            lengths=("uniform", 2, 8), c_ent=0.02),
    "f16_v49152_stream": W["long_seq_grpo"].scaled(n_prompts=1, group=4, T=8, V=49152,
                                                   lengths=("uniform", 2, 8)),
    # the two builds of the loss kernel: rows of at most 100 KB take the short-row one
    # (16 KB chunks: rows of up to 32 KB stay on chip), longer rows the long-row one
    "bf16_v16392_short_stream_min": W["qwen3_0p6b_grpo"].scaled(n_prompts=2, group=4, T=8,
                                                                V=16392, lengths=("uniform", 1, 8),
                                                                c_ent=0.01),
    "bf16_v51200_short_max": W["qwen3_0p6b_grpo"].scaled(n_prompts=2, group=4, T=8, V=51200,
                                                         lengths=("uniform", 1, 8), c_ent=0.01),
    "bf16_v51208_long_min": W["qwen3_0p6b_grpo"].scaled(n_prompts=2, group=4, T=8, V=51208,
                                                        lengths=("uniform", 1, 8), c_ent=0.01),
}
# No masked row: a streamed row's second pass runs in reverse chunk order.
ALL_VALID = {
    "bf16_v151936_long_all_valid": W["ppo_gae"].scaled(n_prompts=8, T=4),
    "bf16_v300001_long_all_valid": W["large_grpo"].scaled(n_prompts=1, group=4, T=4, V=300001,
                                                          lengths=("full",), c_ent=0.0),
    "f32_v100000_long_all_valid": W["tiny_grpo"].scaled(n_prompts=1, group=4, T=4, V=100000,
                                                        lengths=("full",)),
    "f16_v32000_short_all_valid": W["long_seq_grpo"].scaled(n_prompts=1, group=4, T=8,
                                                            lengths=("full",)),
    "f16_v40003_short_all_valid": W["long_seq_grpo"].scaled(n_prompts=1, group=4, T=8, V=40003,
                                                            lengths=("full",), c_ent=0.0,
                                                            beta=0.04),
    "bf16_v16384_short_resident_all_valid": W["qwen3_0p6b_grpo"].scaled(
        n_prompts=2, group=4, T=8, V=16384, lengths=("full",), c_ent=0.01),
}
SMALL.update(ALL_VALID)
PADDED_LD = {"f32_v12345_ragged": 12348, "bf16_v1001_ragged": 1008, "f16_v7_tiny": 8,
             "bf16_v300001_stream": 300008, "bf16_v300001_long_all_valid": 300008,
             "f16_v40003_short_all_valid": 40008}


def _edge_ids(w, chunk_bytes, es, n):
    """Sampled ids on the edges of the ring's chunks and of the row: the first and
    last column, both sides of each chunk boundary, and the last 8 columns."""
    per = chunk_bytes // es
    cols = [0, 1, w.V - 1, w.V - 2]
    for c in range(per, w.V, per):
        cols += [c - 1, c]
    cols += list(range(max(0, w.V - 8), w.V))
    cols = np.array(sorted(set(cols)), dtype=np.int64)
    return cols[np.arange(n) % cols.size]


@pytest.mark.parametrize("name,chunk", [
    ("bf16_v151936_long_all_valid", 32768),   # long-row build, streamed, reverse order
    ("bf16_v300001_stream", 32768),            # long-row build, streamed, load order
    ("f16_v40003_short_all_valid", 16384),     # short-row build, streamed, reverse order
    ("f16_v49152_stream", 16384),              # short-row build, streamed, load order
    ("bf16_v16384_short_resident_all_valid", 16384),  # short-row build, resident rows
])
def test_sampled_id_on_chunk_edges(name, chunk):
    """The sampled logit is read in pass 1 and its -g term written in pass 2 by the
    thread that holds it: ids on every chunk edge, in both pass-2 orders."""
    w = SMALL[name]
    es = {"f32": 4, "bf16": 2, "f16": 2}[w.dtype]
    _run_both(w, ld=PADDED_LD.get(name), ids=_edge_ids(w, chunk, es, w.R))


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
    # rows of at most 100 KB take the short-row build: two CTAs per SM
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert rl.rl_policy_loss_launch_shape("f16", 32000, 1 << 20)[1] == 2 * sms
    assert rl.rl_policy_loss_launch_shape("bf16", 51200, 1 << 20)[1] == 2 * sms
    assert rl.rl_policy_loss_launch_shape("bf16", 51208, 1 << 20)[1] == sms
    assert rl.rl_policy_loss_launch_shape("bf16", 151936, 1 << 20)[1] == sms
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
                                         (5, 0.5, 0.0), (1, 1.0, 0.95), (4096, 1.0, 0.95),
                                         (300, 0.9, 0.99)])
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
    """The benchmark's launch configuration at the workload's full size, at
    grad_scale N and 1: the loss and statistics, logp and entropy of every
    row, every element of every valid row's gradient (the oracle computes
    them on the host a chunk of rows at a time; the comparison runs on the
    device), and every masked row exactly zero."""
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
    d_ids, d_mask = to_dev(ids), to_dev(mask)
    dlogits = torch.empty_like(logits)
    valid = np.nonzero(mask)[0]
    dm = to_dev(mask == 0)
    for gs in (float(N), 1.0):
        out = torch_api.policy_loss(logits, d_ids, d_mask, d_adv, w.B, w.T,
                                    logp_old=to_dev(lo),
                                    ref_logp=to_dev(rf) if rf_arg is not None else None,
                                    eps=w.eps, beta=w.beta, c_ent=w.c_ent, grad_scale=gs,
                                    dlogits=dlogits)
        torch.cuda.synchronize()
        st = torch_api.read_stats(out["stats"])
        assert_stats_match(st, ref, int(band.sum()))
        assert_rows_close(out["logp"].cpu().numpy(), out["entropy"].cpu().numpy(), ref, mask)
        for c0 in range(0, valid.size, 1024):
            sel = valid[c0:c0 + 1024]
            dsel = to_dev(sel)
            host = storage_np(logits.index_select(0, dsel))
            check_dlogits_rows(dlogits.index_select(0, dsel), host, w.dtype, V, ids[sel],
                               np.arange(sel.size), lse[sel], ent[sel], ref_rows(ref, sel),
                               band[sel], np.full(sel.size, gs / N), w.c_ent,
                               where=f"{name} gs={gs:g} rows {sel[0]}..{sel[-1]}")
        for r0 in range(0, R, 4096):  # every masked row is exactly zero
            blk = dlogits[r0:r0 + 4096][dm[r0:r0 + 4096]]
            assert int(torch.count_nonzero(blk.view(torch.int16))) == 0


# ----------------------------------------------------------------- loss options (descriptor API)
def _options_case(seed=7, V=40000, dtype="bf16"):
    w = W["qwen3_0p6b_grpo"].scaled(n_prompts=3, group=4, T=16, V=V, dtype=dtype,
                                    lengths=("uniform", 0, 16), seed=seed, c_ent=0.01)
    small, logits = build_case(w)
    mask = small["mask"].copy()
    mask.reshape(w.B, w.T)[1] = 0          # one empty sequence
    mask.reshape(w.B, w.T)[2, :16] = 1     # one full sequence
    host = storage_np(logits)
    ids = small["ids"]
    lse, logp, ent = oracle.row_stats(host, w.dtype, w.V, ids, mask)
    lo, rf = composed_old_ref(logp, small, mask, w.R)
    return w, small, logits, host, mask, ids, (lse, logp, ent), lo, rf


@pytest.mark.parametrize("agg", ["token_mean", "seq_mean_token_mean", "seq_mean_token_sum",
                                 "token_sum_norm"])
@pytest.mark.parametrize("eps_high", [None, 0.28])
def test_aggregation_and_clip_higher(agg, eps_high):
    w, small, logits, host, mask, ids, (lse, logp, ent), lo, rf = _options_case()
    A = oracle.group_advantages(small["rewards"], w.group)
    arow = np.repeat(A, w.T)
    kw = dict(eps_high=eps_high, agg=agg, T=w.T, agg_norm=100.0)
    ref = oracle.loss_from_stats(logp, ent, mask, arow, lo, rf, w.eps, w.beta, w.c_ent, **kw)
    band = band_mask(ref, w.eps) | (np.abs(ref["r"] - (1 + (eps_high or w.eps))) < CLIP_BAND)
    band &= mask != 0
    gs = 37.0
    out = torch_api.policy_loss(logits, to_dev(ids), to_dev(mask), to_dev(A.astype(np.float32)),
                                w.B, w.T, logp_old=to_dev(lo), ref_logp=to_dev(rf), eps=w.eps,
                                beta=w.beta, c_ent=w.c_ent, grad_scale=gs, eps_high=eps_high,
                                agg=agg, agg_norm=100.0)
    torch.cuda.synchronize()
    st = torch_api.read_stats(out["stats"])
    assert_stats_match(st, ref, int(band.sum()))
    rows = np.arange(w.R)
    check_dlogits_rows(out["dlogits"], host, w.dtype, w.V, ids, rows, lse, ent, ref_rows(ref, rows),
                       band, gs * ref["weights"], w.c_ent, where=agg)


@pytest.mark.parametrize("ddof", [1, 0])
def test_group_rewards_fused_into_the_loss_launch(ddof):
    w, small, logits, host, mask, ids, (lse, logp, ent), lo, rf = _options_case(seed=11, V=8200)
    rewards = to_dev(small["rewards"])
    common = dict(logp_old=to_dev(lo), ref_logp=to_dev(rf), eps=w.eps, beta=w.beta,
                  c_ent=w.c_ent, grad_scale=5.0, agg="seq_mean_token_mean")
    fused = torch_api.policy_loss(logits, to_dev(ids), to_dev(mask), rewards, w.B, w.T,
                                  group_size=w.group, ddof=ddof, **common)
    adv = torch_api.group_advantages(rewards, w.group, ddof=ddof)
    split = torch_api.policy_loss(logits, to_dev(ids), to_dev(mask), adv, w.B, w.T, **common)
    torch.cuda.synchronize()
    # same fp64 arithmetic for the advantages: the two paths agree bit for bit
    assert torch.equal(fused["stats"], split["stats"])
    assert torch.equal(fused["dlogits"].view(torch.int16), split["dlogits"].view(torch.int16))
    # and both match the oracle
    A = oracle.group_advantages(small["rewards"], w.group, ddof=ddof)
    ref = oracle.loss_from_stats(logp, ent, mask, np.repeat(A, w.T), lo, rf, w.eps, w.beta,
                                 w.c_ent, agg="seq_mean_token_mean", T=w.T)
    band = band_mask(ref, w.eps) & (mask != 0)
    assert_stats_match(torch_api.read_stats(fused["stats"]), ref, int(band.sum()))


# ----------------------------------------------------------------- critic
@pytest.mark.parametrize("clip", [None, 0.2])
def test_value_loss_ppo_workload(clip):
    w = W["ppo_gae"]
    small = synth.small_inputs(w)
    _, ret = oracle.gae(small["rewards"], small["values"], small["lengths"], w.gamma, w.lam)
    ret = ret.astype(np.float32).reshape(-1)
    rng = np.random.default_rng(12)
    v = (small["values"].reshape(-1) + rng.normal(0, 0.4, w.R)).astype(np.float32)
    v_old = (small["values"].reshape(-1) + rng.normal(0, 0.4, w.R)).astype(np.float32)
    L = rng.integers(1, w.T + 1, w.B)
    mask = (np.arange(w.T)[None, :] < L[:, None]).astype(np.uint8).reshape(-1)
    N = int(mask.sum())
    ref = oracle.value_loss(v, v_old if clip else None, ret, mask, clip, grad_scale=N)
    dv, st = torch_api.value_loss(to_dev(v), to_dev(ret), to_dev(mask),
                                  values_old=to_dev(v_old) if clip else None,
                                  clip_eps=clip if clip else -1.0, grad_scale=float(N))
    dv = dv.cpu().numpy()
    # tokens at a kink (clip boundary or equal squares) may take either branch
    vd, vo64, r64 = v.astype(np.float64), v_old.astype(np.float64), ret.astype(np.float64)
    if clip:
        vc = vo64 + np.clip(vd - vo64, -clip, clip)
        kink = (np.abs(np.abs(vd - vo64) - clip) < 1e-5) | (np.abs((vc - r64) ** 2 - (vd - r64) ** 2) < 1e-5)
    else:
        kink = np.zeros(w.R, bool)
    kink &= mask != 0
    assert st["n_tokens"] == N
    assert abs(st["n_clipped"] - ref["n_clipped"]) <= int(kink.sum())
    assert_scalar_close("value loss", st["loss"], ref["loss"])
    assert_scalar_close("mean_abs_err", st["mean_abs_err"], ref["mean_abs_err"])
    ok = ~kink
    np.testing.assert_allclose(dv[ok], ref["dvalues"][ok], rtol=1e-5, atol=1e-6)
    assert np.all(dv[mask == 0] == 0)


# ----------------------------------------------------------------- autograd and CUDA graphs
def _small_inputs_dev(name="qwen_vocab_bf16_c2"):
    w = SMALL[name]
    small, logits = build_case(w)
    return w, small, logits, to_dev(small["ids"]), to_dev(small["mask"]), to_dev(small["rewards"])


def test_autograd_function_matches_direct_call():
    w, small, logits, ids, mask, rewards = _small_inputs_dev()
    opts = dict(eps=w.eps, c_ent=0.01, group_size=w.group, agg="seq_mean_token_mean")
    direct = torch_api.policy_loss(logits, ids, mask, rewards, w.B, w.T, **opts)
    x = logits.clone().requires_grad_(True)
    loss, logp, ent = torch_api.FusedPolicyLoss.apply(x, ids, mask, rewards, w.B, w.T, opts)
    (3.0 * loss).backward()
    st = torch_api.read_stats(direct["stats"])
    assert float(loss.detach()) == st["loss"]
    assert torch.equal(logp, direct["logp"]) and torch.equal(ent, direct["entropy"])
    expect = direct["dlogits"] * torch.tensor(3.0, dtype=logits.dtype, device=logits.device)
    assert torch.equal(x.grad.view(torch.int16), expect.view(torch.int16))


def test_cuda_graph_capture_replays_the_step():
    w, small, logits, ids, mask, rewards = _small_inputs_dev()
    adv = torch.empty(w.B, device="cuda")
    dl = torch.empty_like(logits)
    lp = torch.empty(w.R, device="cuda")
    en = torch.empty(w.R, device="cuda")
    ws = torch_api.new_workspace(w.R, "cuda")
    st = torch_api.new_stats("cuda")

    def step(s=None):
        torch_api.group_advantages(rewards, w.group, out=adv, stream=s)
        torch_api.policy_loss(logits, ids, mask, adv, w.B, w.T, eps=w.eps, c_ent=0.01,
                              grad_scale=9.0, dlogits=dl, logp_out=lp, entropy_out=en,
                              workspace=ws, stats=st, stream=s)

    step()  # warm-up: launch plans are cached before capture
    torch.cuda.synchronize()
    eager = (dl.clone(), st.clone(), lp.clone())
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            step(s)
    dl.zero_()
    st.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(dl.view(torch.int16), eager[0].view(torch.int16))
    assert torch.equal(st, eager[1]) and torch.equal(lp, eager[2])
    # new inputs in the same buffers: the replay follows them
    logits.mul_(0.5)
    g.replay()
    torch.cuda.synchronize()
    replayed = (dl.clone(), st.clone())
    step()
    torch.cuda.synchronize()
    assert torch.equal(dl.view(torch.int16), replayed[0].view(torch.int16))
    assert torch.equal(st, replayed[1])


# ----------------------------------------------------------------- whitening
@pytest.mark.parametrize("shift", [True, False])
def test_masked_whiten_ppo_advantages(shift):
    w = W["ppo_gae"]
    small = synth.small_inputs(w)
    A, _ = oracle.gae(small["rewards"], small["values"], small["lengths"], w.gamma, w.lam)
    A = A.astype(np.float32).reshape(-1)
    rng = np.random.default_rng(13)
    L = rng.integers(0, w.T + 1, w.B)
    mask = (np.arange(w.T)[None, :] < L[:, None]).astype(np.uint8).reshape(-1)
    ref = oracle.masked_whiten(A, mask, 1e-8, shift)
    d = to_dev(A)
    got = torch_api.masked_whiten(d, to_dev(mask), 1e-8, shift).cpu().numpy()
    assert np.all(np.abs(got - ref) <= ADV_TOL * np.maximum(np.abs(ref), 1.0))
    torch_api.masked_whiten(d, to_dev(mask), 1e-8, shift, out=d)  # in place
    assert np.array_equal(d.cpu().numpy(), got)


@pytest.mark.parametrize("n", [1, 7, 1000, 8192, 8193, 100003])
def test_masked_whiten_sizes(n):
    """Sizes around the kernel's 8192-element step (1024 threads x 8), a lone
    element and a ragged large case."""
    rng = np.random.default_rng(n)
    x = rng.normal(0.3, 2.0, n).astype(np.float32)
    mask = (rng.random(n) < 0.7).astype(np.uint8)
    ref = oracle.masked_whiten(x, mask, 1e-8, True)
    got = torch_api.masked_whiten(to_dev(x), to_dev(mask), 1e-8, True).cpu().numpy()
    assert np.all(np.abs(got - ref) <= ADV_TOL * np.maximum(np.abs(ref), 1.0))


@pytest.mark.parametrize("n", [1, 8193, 100003])
def test_value_loss_sizes(n):
    rng = np.random.default_rng(n + 1)
    v = rng.normal(0, 1, n).astype(np.float32)
    vo = (v + rng.normal(0, 0.3, n)).astype(np.float32)
    ret = rng.normal(0, 1, n).astype(np.float32)
    mask = (rng.random(n) < 0.6).astype(np.uint8)
    N = int(mask.sum())
    ref = oracle.value_loss(v, vo, ret, mask, 0.2, grad_scale=max(N, 1))
    dv, st = torch_api.value_loss(to_dev(v), to_dev(ret), to_dev(mask), values_old=to_dev(vo),
                                  clip_eps=0.2, grad_scale=float(max(N, 1)))
    assert st["n_tokens"] == N
    assert abs(st["loss"] - ref["loss"]) <= LOSS_RTOL * max(abs(ref["loss"]), 1e-3)
    # tokens at a kink (clip boundary or equal squares) may take either branch
    vd, vo64, r64 = v.astype(np.float64), vo.astype(np.float64), ret.astype(np.float64)
    vc = vo64 + np.clip(vd - vo64, -0.2, 0.2)
    kink = (np.abs(np.abs(vd - vo64) - 0.2) < 1e-5) | (np.abs((vc - r64) ** 2 - (vd - r64) ** 2) < 1e-5)
    ok = ~kink
    got = dv.cpu().numpy()
    assert np.all(np.abs(got - ref["dvalues"])[ok] <= 1e-5 * np.maximum(np.abs(ref["dvalues"]), 1.0)[ok])


# ----------------------------------------------------------------- randomized sweep
def _random_case(seed):
    rng = np.random.default_rng(1000 + seed)
    dtype = ["f32", "bf16", "f16"][rng.integers(0, 3)]
    es = {"f32": 4, "bf16": 2, "f16": 2}[dtype]
    u = rng.random()
    V = (int(rng.choice([1, 2, 3, 7, 8, 9, 63, 64, 65])) if u < 0.4 else
         int(rng.integers(1, 5001)) if u < 0.8 else int(rng.integers(50000, 120001)))
    align = 16 // es
    ld = -(-V // align) * align + align * int(rng.integers(0, 3))
    G = int(rng.integers(1, 4))
    n_prompts = int(rng.integers(1, 4))
    T = int(rng.integers(1, 12))
    style = rng.integers(0, 4)
    lengths = ("uniform", 0, 0) if style == 0 else ("full",) if style == 1 else ("uniform", 0, T)
    w = W["tiny_grpo"].scaled(dtype=dtype, V=V, group=G + 1, n_prompts=n_prompts, T=T,
                              lengths=lengths, seed=2000 + seed,
                              c_ent=float(rng.choice([0.0, 0.03])),
                              beta=float(rng.choice([0.0, 0.05])))
    opts = dict(with_old=bool(rng.integers(0, 2)), in_place=bool(rng.integers(0, 2)),
                agg=str(rng.choice(oracle.AGGREGATIONS)),
                eps_high=float(rng.choice([-1.0, 0.3])))
    return w, ld, opts


@pytest.mark.parametrize("seed", range(24))
def test_randomized_shapes_and_options(seed):
    w, ld, o = _random_case(seed)
    small, logits = build_case(w, ld=ld)
    V, R = w.V, w.R
    mask, ids = small["mask"], small["ids"]
    A = oracle.group_advantages(small["rewards"], w.group)
    arow = np.repeat(A, w.T)
    host = storage_np(logits)[:, :V]
    lse, logp, ent = oracle.row_stats(host, w.dtype, V, ids, mask)
    lo, rf = composed_old_ref(logp, small, mask, R)
    eps_high = None if o["eps_high"] < 0 else o["eps_high"]
    ref = oracle.loss_from_stats(logp, ent, mask, arow, lo if o["with_old"] else None,
                                 rf if w.beta else None, w.eps, w.beta, w.c_ent, eps_high=eps_high,
                                 agg=o["agg"], T=w.T, agg_norm=50.0)
    band = (band_mask(ref, w.eps) | (np.abs(ref["r"] - (1 + (eps_high or w.eps))) < CLIP_BAND)) & (mask != 0)
    N = ref["n_tokens"]
    gs = float(max(N, 1))
    src = logits.clone() if o["in_place"] else logits
    dst = src if o["in_place"] else torch.full_like(logits, 7.0)
    out = torch_api.policy_loss(src, to_dev(ids), to_dev(mask), to_dev(A.astype(np.float32)),
                                w.B, w.T, V=V, logp_old=to_dev(lo) if o["with_old"] else None,
                                ref_logp=to_dev(rf) if w.beta else None, eps=w.eps, beta=w.beta,
                                c_ent=w.c_ent, grad_scale=gs, dlogits=dst, eps_high=eps_high,
                                agg=o["agg"], agg_norm=50.0)
    torch.cuda.synchronize()
    st = torch_api.read_stats(out["stats"])
    assert_stats_match(st, ref, int(band.sum()))
    assert_rows_close(out["logp"].cpu().numpy(), out["entropy"].cpu().numpy(), ref, mask)
    rows = np.arange(R)
    check_dlogits_rows(out["dlogits"][:, :V], host, w.dtype, V, ids, rows, lse, ent,
                       ref_rows(ref, rows), band, gs * ref["weights"], w.c_ent,
                       where=f"seed {seed} {w.dtype} V={V} ld={ld} {o}")
    if ld != V and not o["in_place"]:
        assert bool((out["dlogits"][:, V:] == 7.0).all())


# ----------------------------------------------------------------- data parallelism
@pytest.mark.parametrize("agg", ["token_mean", "seq_mean_token_mean", "seq_mean_token_sum"])
def test_global_counts_split_batch(agg):
    w = W["qwen3_0p6b_grpo"].scaled(n_prompts=2, group=4, T=16, V=40000,
                                    lengths=("uniform", 0, 16), c_ent=0.01)
    small, logits = build_case(w)
    mask = small["mask"].copy()
    mask.reshape(w.B, w.T)[2] = 0
    m_d, ids_d = to_dev(mask), to_dev(small["ids"])
    adv_d = to_dev(oracle.group_advantages(small["rewards"], w.group).astype(np.float32))
    counts = torch_api.count_tokens(m_d, w.B, w.T)
    L = mask.reshape(w.B, w.T).sum(1)
    assert counts.tolist() == [int(mask.sum()), int((L > 0).sum())]
    kw = dict(eps=w.eps, c_ent=w.c_ent, grad_scale=3.0, agg=agg)
    full = torch_api.policy_loss(logits, ids_d, m_d, adv_d, w.B, w.T, **kw)
    h = w.B // 2
    halves = [torch_api.policy_loss(logits[s * h * w.T:(s + 1) * h * w.T], ids_d[s * h * w.T:(s + 1) * h * w.T],
                                    m_d[s * h * w.T:(s + 1) * h * w.T], adv_d[s * h:(s + 1) * h], h, w.T,
                                    global_counts=counts, **kw) for s in range(2)]
    torch.cuda.synchronize()
    st = torch_api.read_stats(full["stats"])
    parts = [torch_api.read_stats(x["stats"]) for x in halves]
    for k in ("loss", "pg_term", "ent_term", "clip_frac"):
        assert_scalar_close(k, parts[0][k] + parts[1][k], st[k])
    assert parts[0]["n_tokens"] + parts[1]["n_tokens"] == st["n_tokens"]
    cat = torch.cat([x["dlogits"] for x in halves])
    assert torch.equal(cat.view(torch.int16), full["dlogits"].view(torch.int16))


def test_loss_waits_for_the_kernel_before_it():
    """The loss launch may start while the kernel before it in the stream still
    runs (programmatic dependent launch); it must still read that kernel's
    output.  A single-CTA whitening over a long buffer (the advantages plus
    four million masked-out elements, ~1 ms) rewrites the per-token
    advantages in place, and the loss is launched right after it with no host
    synchronisation: the loss must match the oracle on the WHITENED
    advantages."""
    w = W["ppo_gae"].scaled(n_prompts=8)
    small = synth.small_inputs(w)
    logits = synth.logits(w, device="cuda")
    V, R = w.V, w.R
    mask, ids = small["mask"], small["ids"]
    A, _ = oracle.gae(small["rewards"], small["values"], small["lengths"], w.gamma, w.lam)
    A = A.astype(np.float32).reshape(-1)
    extra = 4 << 20
    buf = np.concatenate([A, np.full(extra, 123.0, np.float32)])
    wmask = np.concatenate([mask, np.zeros(extra, np.uint8)])
    A_w = oracle.masked_whiten(A, mask, 1e-8, True).astype(np.float32)
    lse, logp, ent = oracle_stats_chunked(logits, w.dtype, V, ids, mask)
    lo, _ = composed_old_ref(logp, small, mask, R)
    ref = oracle.loss_from_stats(logp, ent, mask, A_w.astype(np.float64), lo, None, w.eps, 0.0,
                                 w.c_ent)
    band = band_mask(ref, w.eps) & (mask != 0)
    d_buf, d_wmask = to_dev(buf), to_dev(wmask)
    d_ids, d_mask, d_lo = to_dev(ids), to_dev(mask), to_dev(lo)
    torch.cuda.synchronize()
    torch_api.masked_whiten(d_buf, d_wmask, 1e-8, True, out=d_buf)  # in place, ~1 ms
    out = torch_api.policy_loss(logits, d_ids, d_mask, d_buf[:R], w.B, w.T, logp_old=d_lo,
                                eps=w.eps, beta=0.0, c_ent=w.c_ent, grad_scale=1.0,
                                dlogits=None)
    torch.cuda.synchronize()
    assert np.all(np.abs(d_buf[:R].cpu().numpy() - A_w) <= ADV_TOL * np.maximum(np.abs(A_w), 1.0))
    assert_stats_match(torch_api.read_stats(out["stats"]), ref, int(band.sum()))


@pytest.mark.parametrize("V", [9, 32000, 151936])
def test_rows_at_the_fp16_floor(V):
    """Rows whose every logit is -65504, the lowest finite fp16 value: a
    uniform distribution, logp = -ln V and entropy ln V.  In the vector that a
    row's end cuts, the first pass sets the elements past the end to the
    format's floor (-65504 in fp16), and only in rows whose maximum is that
    floor do they reach the softmax sums; the kernel takes their share out
    again.  At V = 9 (a 16-element row stride) those are 7 elements, and
    without the correction the row would read as uniform over 16 (logp off by
    0.58).  V = 32000 (short-row build) and 151936 (long-row build) end on a
    vector boundary and have partly filled last chunks.  At |z| = 65504 fp32
    resolves about 2^-8 in any implementation, so these rows are checked to
    1e-2; every other row to the usual tolerance."""
    w = W["long_seq_grpo"].scaled(dtype="f16", V=V, n_prompts=1, group=4, T=4,
                                  lengths=("full",), c_ent=0.02, beta=0.05, seed=91)
    ld = -(-V // 8) * 8
    small, logits = build_case(w, ld=ld)
    R = w.R
    ids = small["ids"].copy()
    floor_rows = [1, 6]
    for r in floor_rows:
        logits[r, :V] = -65504.0
    host = storage_np(logits)[:, :V]
    mask = small["mask"]
    assert mask.all()
    arow, adv = adv_rows(w, small)
    lse, logp, ent = oracle.row_stats(host, "f16", V, ids, mask)
    lo, rf = composed_old_ref(logp, small, mask, R)
    out = torch_api.policy_loss(logits, to_dev(ids), to_dev(mask), to_dev(adv.astype(np.float32)),
                                w.B, w.T, V=V, logp_old=to_dev(lo), ref_logp=to_dev(rf), eps=w.eps,
                                beta=w.beta, c_ent=w.c_ent, grad_scale=1.0)
    torch.cuda.synchronize()
    lp_gpu = out["logp"].cpu().numpy()
    h_gpu = out["entropy"].cpu().numpy()
    for r in floor_rows:
        assert abs(logp[r] + np.log(V)) < 1e-9 and abs(ent[r] - np.log(V)) < 1e-9  # the oracle
        assert abs(lp_gpu[r] + np.log(V)) < 1e-2, (r, lp_gpu[r], -np.log(V))
        assert abs(h_gpu[r] - np.log(V)) < 1e-2, (r, h_gpu[r], np.log(V))
    keep = np.ones(R, dtype=bool)
    keep[floor_rows] = False
    assert np.abs(lp_gpu[keep] - logp[keep]).max() <= LOGP_ATOL
    assert np.abs(h_gpu[keep] - ent[keep]).max() <= LOGP_ATOL
    assert not torch.isnan(out["dlogits"][:, :V].float()).any()


@pytest.mark.parametrize("dtype,V", [("bf16", 151936), ("f16", 32000), ("f32", 5000)])
def test_minus_infinity_and_extreme_logits(dtype, V):
    """Padded-vocabulary rows: the last 267 entries of every row are -inf (as
    when a 151,669-token vocabulary is padded to 151,936), 1% of the other
    entries are -inf, and a few rows carry extreme logits (+3e4 and -3e4 in
    16-bit formats, 1e6 in fp32: a max far from the bulk, exponents that
    underflow; one row scaled by 10).  Sampled ids
    are finite entries.  With the entropy bonus and the KL term on, every
    output must match the oracle, which takes 0 log 0 = 0."""
    base = W["qwen3_0p6b_grpo"] if dtype == "bf16" else W["long_seq_grpo"]
    w = base.scaled(dtype=dtype, V=V, n_prompts=2, group=4, T=6, lengths=("uniform", 1, 6),
                    c_ent=0.02, beta=0.05, seed=77)
    small = synth.small_inputs(w)
    logits = synth.logits(w, device="cuda")
    R = w.R
    g = torch.Generator(device="cuda").manual_seed(5)
    hole = torch.rand((R, V), generator=g, device="cuda") < 0.01
    hole[:, V - 267:] = True
    logits[hole] = float("-inf")
    big = 3e4 if dtype != "f32" else 1e6
    logits[1, 10] = big
    logits[2, 11] = -big
    logits[3, ::7] = logits[3, ::7] * 10.0
    host = storage_np(logits)
    zf = oracle.decode(host, dtype)
    ids = small["ids"].copy()
    for r in range(R):  # a sampled token has a finite logit
        while not np.isfinite(zf[r, ids[r]]):
            ids[r] = (ids[r] + 1) % (V - 267)
    # row 1 samples its dominant entry (logp ~ 0); a sampled logp near -3e4 would leave fp32
    # too few bits for the ratio exp(logp - logp_old), in any implementation
    ids[1] = 10
    mask = small["mask"]
    arow, adv = adv_rows(w, small)
    lse, logp, ent = oracle.row_stats(host, dtype, V, ids, mask)
    lo, rf = composed_old_ref(logp, small, mask, R)
    ref = oracle.loss_from_stats(logp, ent, mask, arow, lo, rf, w.eps, w.beta, w.c_ent)
    band = band_mask(ref, w.eps) & (mask != 0)
    N = ref["n_tokens"]
    out = torch_api.policy_loss(logits, to_dev(ids), to_dev(mask), to_dev(adv.astype(np.float32)),
                                w.B, w.T, logp_old=to_dev(lo), ref_logp=to_dev(rf), eps=w.eps,
                                beta=w.beta, c_ent=w.c_ent, grad_scale=float(N))
    torch.cuda.synchronize()
    st = torch_api.read_stats(out["stats"])
    assert_stats_match(st, ref, int(band.sum()))
    assert_rows_close(out["logp"].cpu().numpy(), out["entropy"].cpu().numpy(), ref, mask)
    rows = np.arange(R)
    scale = np.where(mask != 0, 1.0, 0.0)  # grad_scale N times the 1/N of the token mean
    check_dlogits_rows(out["dlogits"], host, dtype, V, ids, rows, lse, ent, ref_rows(ref, rows),
                       band, scale, w.c_ent, where=f"{dtype} V={V}")
    assert not torch.isnan(out["dlogits"].float()).any()
