"""GPU parity of rl_lmhead_logprobs (the LM-head projection fused with the
row log-softmax statistics, on the tensor cores) against the fp64 oracle:
the exact product of the bf16 inputs, then lse, log-prob of the sampled id
and entropy per row.

Tolerance: the kernel accumulates the exact bf16 products in fp32, so each
logit carries an absolute error of at most about D * 2^-24 * sum|h_d w_vd|
(a few 1e-6 here); the row statistics then follow the policy-loss kernel's
fp32 arithmetic, whose bound is LOGP_ATOL (2e-3 absolute) on lse, logp and
entropy.  Small cases compare every row; the full Qwen3 LM-head shape
(D = 1024, V = 151936) compares sampled rows.
"""
import numpy as np
import pytest
import torch

import oracle
import ppo_policy_loss_gb300 as rl
from ppo_policy_loss_gb300 import synth
from _parity import LOGP_ATOL, storage_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    rl.build()
    rl.load()


def run_gpu(hidden, weight, ids, D, V, status=None, sliced=True, ws_bytes=None, dev_inputs=None):
    """Run the kernel; with ``sliced`` the call gets a zeroed workspace (of
    ``ws_bytes``, default the library's size for this shape), which it must
    leave zeroed again."""
    dev = torch.device("cuda:0")
    h, w, i = dev_inputs if dev_inputs is not None else (hidden.to(dev), weight.to(dev), ids.to(dev))
    R = h.shape[0]
    dtype = "f16" if h.dtype == torch.float16 else "bf16"
    lse = torch.full((R,), 7.0, device=dev)
    logp = torch.full((R,), 7.0, device=dev)
    ent = torch.full((R,), 7.0, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev) if status is None else status
    ws = None
    if sliced:
        nb = rl.rl_lmhead_workspace_size(R, V) if ws_bytes is None else ws_bytes
        ws = torch.zeros(max(nb, 16), dtype=torch.uint8, device=dev)
    rl.rl_lmhead_logprobs(h, h.stride(0), w, w.stride(0), dtype, R, D, V, i, logp, ent, lse, st,
                          ws, ws.numel() if ws is not None else 0)
    torch.cuda.synchronize()
    if ws is not None and rl.rl_lmhead_plan(R, D, V, ws.numel())[0] > 1:
        n_mt = -(-R // 128)
        assert int(ws[: n_mt * 4].view(torch.int32).abs().sum()) == 0, "tickets not reset"
    return lse.cpu().numpy(), logp.cpu().numpy(), ent.cpu().numpy(), int(st.item())


def oracle_rows(hidden, weight, ids, D, rows=None):
    h = storage_np(hidden)[:, :D]
    w = storage_np(weight)[:, :D]
    idn = ids.numpy()
    if rows is not None:
        h, idn = h[rows], idn[rows]
    return oracle.lmhead_row_stats(h, w, idn, "f16" if hidden.dtype == torch.float16 else "bf16")


def check(got, ref, rows=slice(None)):
    for name, g, r in zip(("lse", "logp", "entropy"), got, ref):
        g = g[rows]
        assert np.isfinite(g).all(), name
        err = np.abs(g.astype(np.float64) - r)
        assert err.max() <= LOGP_ATOL, (name, float(err.max()), int(err.argmax()))


@pytest.mark.parametrize("sliced", [False, True])
@pytest.mark.parametrize("R,D,V,ld_h,ld_w,sd,seed", [
    (128, 64, 256, None, None, 2.0, 1),          # one tile
    (128, 128, 512, None, None, 2.0, 2),         # two K blocks, two N tiles
    (300, 200, 1000, 208, 256, 2.0, 3),          # ragged R, D (zero-filled K tail), V; padded strides
    (1, 8, 1, None, None, 1.0, 4),               # the smallest shape
    (257, 64, 33, None, None, 8.0, 5),           # V below one tile, wide logits
    (640, 256, 4096, None, None, 12.0, 6),       # running-max rescales across tiles
])
def test_lmhead_small(R, D, V, ld_h, ld_w, sd, seed, sliced):
    hidden, weight, ids = synth.lmhead_inputs(R, D, V, seed, sd, ld_h, ld_w)
    lse, logp, ent, st = run_gpu(hidden, weight, ids, D, V, sliced=sliced)
    assert st == 0
    check((lse, logp, ent), oracle_rows(hidden, weight, ids, D))


@pytest.mark.parametrize("sliced", [False, True])
def test_lmhead_persistent_tiles(sliced):
    """More 128-row tiles than SMs: CTAs loop over units and reuse both
    tensor-memory accumulators."""
    R = 128 * 330 + 17
    hidden, weight, ids = synth.lmhead_inputs(R, 128, 768, 7, 3.0)
    lse, logp, ent, st = run_gpu(hidden, weight, ids, 128, 768, sliced=sliced)
    assert st == 0
    check((lse, logp, ent), oracle_rows(hidden, weight, ids, 128))


def test_lmhead_slice_counts_agree():
    """Workspaces that cap the split at different slice counts (1, 2, 3 and
    the library's choice) give the oracle's statistics on every row, and a
    repeated call with one workspace is bitwise identical (the partials are
    merged in slice order, whatever order the units finish in)."""
    R, D, V = 1000, 256, 151936 // 4
    hidden, weight, ids = synth.lmhead_inputs(R, D, V, 11, 3.0)
    ref = oracle_rows(hidden, weight, ids, D)
    dev = torch.device("cuda:0")
    dev_in = (hidden.to(dev), weight.to(dev), ids.to(dev))
    n_mt = -(-R // 128)
    seen = set()
    for k in (1, 2, 3, None):
        nb = None if k is None else ((n_mt * 4 + 255) // 256 * 256 + k * R * 16 if k > 1 else 0)
        ns = rl.rl_lmhead_plan(R, D, V, rl.rl_lmhead_workspace_size(R, V) if nb is None else nb)[0]
        seen.add(ns)
        got = run_gpu(None, None, None, D, V, ws_bytes=nb, dev_inputs=dev_in)
        assert got[3] == 0
        check(got[:3], ref)
        again = run_gpu(None, None, None, D, V, ws_bytes=nb, dev_inputs=dev_in)
        for a_, b_ in zip(got[:3], again[:3]):
            assert np.array_equal(a_, b_)
    assert len(seen) >= 3, seen


def test_lmhead_qwen3_shape_sampled_rows():
    """The Qwen3-0.6B LM head (D 1024, V 151936) on 32 x 1024 rows; the
    oracle recomputes 96 sampled rows, including the first and last."""
    R, D, V = 32 * 1024, 1024, 151936
    hidden, weight, ids = synth.lmhead_inputs(R, D, V, 8, 3.0)
    assert rl.rl_lmhead_plan(R, D, V, rl.rl_lmhead_workspace_size(R, V))[0] > 1
    lse, logp, ent, st = run_gpu(hidden, weight, ids, D, V)
    assert st == 0
    assert np.isfinite(lse).all() and np.isfinite(logp).all() and np.isfinite(ent).all()
    rng = np.random.default_rng(8)
    rows = np.unique(np.concatenate([[0, R - 1], rng.choice(R, 94, replace=False)]))
    ref = oracle_rows(hidden, weight, ids, D, rows)
    check((lse[rows], logp[rows], ent[rows]), ref)
    # logp <= 0 and 0 <= H <= log V hold for every row
    assert (logp <= 1e-5).all() and (ent >= -1e-5).all() and (ent <= np.log(V) + 1e-4).all()


def test_lmhead_bad_id_sets_status():
    hidden, weight, ids = synth.lmhead_inputs(130, 64, 300, 9)
    ids[5] = 300
    ids[129] = -1
    lse, logp, ent, st = run_gpu(hidden, weight, ids, 64, 300)
    assert st & rl.RL_DEVERR_ID_RANGE
    assert np.isnan(logp[5]) and np.isnan(logp[129])
    good = np.setdiff1d(np.arange(130), [5, 129])
    ids_ok = ids.clone()
    ids_ok[5] = 0
    ids_ok[129] = 0
    ref = oracle_rows(hidden, weight, ids_ok, 64)
    check((lse, logp, ent), [r[good] for r in ref], good)


def test_lmhead_optional_outputs_and_empty():
    hidden, weight, ids = synth.lmhead_inputs(200, 64, 500, 10)
    dev = torch.device("cuda:0")
    h, w, i = hidden.to(dev), weight.to(dev), ids.to(dev)
    logp = torch.empty(200, device=dev)
    rl.rl_lmhead_logprobs(h, 64, w, 64, "bf16", 200, 64, 500, i, logp, None, None, None)
    torch.cuda.synchronize()
    ref = oracle_rows(hidden, weight, ids, 64)
    assert np.abs(logp.cpu().numpy() - ref[1]).max() <= LOGP_ATOL
    rl.rl_lmhead_logprobs(h, 64, w, 64, "bf16", 0, 64, 500, i, logp, None, None, None)  # R = 0: no launch
    torch.cuda.synchronize()


@pytest.mark.parametrize("case", range(12))
def test_lmhead_randomized(case):
    """Seeded random shapes: R in [1, 3000], D a multiple of 8 in [8, 520]
    (ragged K tails), V in [1, 5000], padded strides, logit spreads 0.5-12,
    with and without a workspace."""
    rng = np.random.default_rng(1000 + case)
    R = int(rng.integers(1, 3001))
    D = int(rng.integers(1, 66)) * 8
    V = int(rng.integers(1, 5001))
    ld_h = D + 8 * int(rng.integers(0, 3))
    ld_w = D + 8 * int(rng.integers(0, 3))
    sd = float(rng.uniform(0.5, 12.0))
    hidden, weight, ids = synth.lmhead_inputs(R, D, V, 2000 + case, sd, ld_h, ld_w)
    got = run_gpu(hidden, weight, ids, D, V, sliced=bool(case % 2))
    assert got[3] == 0
    check(got[:3], oracle_rows(hidden, weight, ids, D))


@pytest.mark.parametrize("sliced", [False, True])
def test_lmhead_unit_groups(sliced):
    """D = 4096 (the Qwen3-8B head's hidden size) puts 40 row tiles in a unit
    group, so 45 row tiles make a full group and a 5-tile tail group."""
    R, D, V = 128 * 45 - 3, 4096, 3000
    ws_bytes = rl.rl_lmhead_workspace_size(R, V) if sliced else 0
    plan = rl.rl_lmhead_plan(R, D, V, ws_bytes)
    assert plan[2] == 40 and (plan[0] > 1) == sliced
    hidden, weight, ids = synth.lmhead_inputs(R, D, V, 12, 4.0)
    got = run_gpu(hidden, weight, ids, D, V, sliced=sliced)
    assert got[3] == 0
    check(got[:3], oracle_rows(hidden, weight, ids, D))


def test_lmhead_torch_api_and_cuda_graph():
    """torch_api.lmhead_logprobs matches the oracle, and the launch captured in a
    CUDA graph replays to the same bits (the tensor maps travel as launch
    parameters; the workspace tickets are left at zero by every launch)."""
    from ppo_policy_loss_gb300 import torch_api
    R, D, V = 1000, 256, 20000
    hidden, weight, ids = synth.lmhead_inputs(R, D, V, 21, 3.0)
    dev = torch.device("cuda:0")
    h, w, i = hidden.to(dev), weight.to(dev), ids.to(dev)
    out = torch_api.lmhead_logprobs(h, w, i, want_lse=True)
    torch.cuda.synchronize()
    check((out["lse"].cpu().numpy(), out["logp"].cpu().numpy(), out["entropy"].cpu().numpy()),
          oracle_rows(hidden, weight, ids, D))
    ws = out["workspace"]
    lp = torch.empty(R, device=dev)
    s = torch.cuda.Stream(dev)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            rl.rl_lmhead_logprobs(h, D, w, D, "bf16", R, D, V, i, lp, None, None, None, ws,
                                  ws.numel() if ws is not None else 0, s)
    for _ in range(3):
        lp.fill_(7.0)
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(lp, out["logp"])


def test_lmhead_zero_hidden_rows_are_uniform():
    """A zero hidden state gives all-zero logits: lse = entropy = ln V and
    logp = -ln V exactly in closed form (the uniform distribution)."""
    R, D, V = 300, 128, 151936
    hidden, weight, ids = synth.lmhead_inputs(R, D, V, 23, 3.0)
    zero = np.arange(0, R, 7)
    hidden[zero] = 0
    lse, logp, ent, st = run_gpu(hidden, weight, ids, D, V)
    assert st == 0
    lnV = np.log(V)
    assert np.abs(lse[zero] - lnV).max() <= LOGP_ATOL
    assert np.abs(ent[zero] - lnV).max() <= LOGP_ATOL
    assert np.abs(logp[zero] + lnV).max() <= LOGP_ATOL
    check((lse, logp, ent), oracle_rows(hidden, weight, ids, D))


@pytest.mark.parametrize("R,D,V,sliced", [(300, 200, 1000, False), (1000, 1024, 30000, True)])
def test_lmhead_fp16_inputs(R, D, V, sliced):
    """fp16 hidden states and weight (the pages' FP16 inputs with FP32
    accumulation): the same kernel with fp16 tensor-core operands."""
    hidden, weight, ids = synth.lmhead_inputs(R, D, V, 31 + R, 3.0)
    hidden, weight = hidden.float().half(), weight.float().half()  # bf16 values are exact in fp16 here
    lse, logp, ent, st = run_gpu(hidden, weight, ids, D, V, sliced=sliced)
    assert st == 0
    check((lse, logp, ent), oracle_rows(hidden, weight, ids, D))
