"""CPU-side checks of the C ABI: the library builds for sm_103a, loads, exports
every function include/rlloss.h declares, and rejects bad arguments on the
host before anything is launched (no GPU needed; fake device addresses are
never dereferenced on these paths)."""
import ctypes
import os
import re
import shutil
import subprocess

import pytest

import ppo_policy_loss_gb300 as rl

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "rlloss.h")

pytestmark = pytest.mark.skipif(shutil.which("nvcc") is None and not os.path.exists(
    "/usr/local/cuda/bin/nvcc"), reason="no CUDA toolkit")


@pytest.fixture(scope="module")
def lib():
    rl.build()
    return rl.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(rl_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("rl_group_advantages", "rl_gae_reverse_scan", "rl_policy_loss_fwd_bwd",
              "rl_policy_loss_workspace_size", "rl_read_device_status", "rl_status_string",
              "rl_policy_loss_launch_shape"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", rl.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\bT\s+(\w+)", out))
    for n in declared_functions():
        assert n in exported, n
        assert hasattr(lib, n)


def test_status_strings(lib):
    for s in range(11):
        assert rl.rl_status_string(s) and rl.rl_status_string(s) != "unknown status"
    assert rl.rl_status_string(99) == "unknown status"


def test_workspace_size(lib):
    n = rl.rl_policy_loss_workspace_size(131072)
    assert n >= 256 and n % 16 == 0
    assert rl.rl_policy_loss_workspace_size(0) == n


FAKE = 0x7F0000000000  # 16-byte aligned, never dereferenced on error paths


def call_loss(lib, **over):
    a = dict(logits=FAKE, dtype=rl.RL_BF16, B=2, T=4, V=1024, ld=1024, ids=FAKE + 0x100000,
             logp_old=None, ref_logp=None, mask=FAKE + 0x200000, adv=FAKE + 0x300000,
             adv_layout=rl.RL_ADV_PER_SEQ, eps=0.2, beta=0.0, c_ent=0.0, grad_scale=1.0,
             dlogits=FAKE + 0x400000, logp_out=None, entropy_out=None, stats=FAKE + 0x500000,
             workspace=FAKE + 0x600000, ws_bytes=rl.rl_policy_loss_workspace_size(8), stream=None)
    a.update(over)
    return lib.rl_policy_loss_fwd_bwd(a["logits"], a["dtype"], a["B"], a["T"], a["V"], a["ld"],
                                      a["ids"], a["logp_old"], a["ref_logp"], a["mask"], a["adv"],
                                      a["adv_layout"], a["eps"], a["beta"], a["c_ent"],
                                      a["grad_scale"], a["dlogits"], a["logp_out"],
                                      a["entropy_out"], a["stats"], a["workspace"], a["ws_bytes"],
                                      a["stream"])


@pytest.mark.parametrize("over,status", [
    (dict(dtype=7), rl.RL_ERR_DTYPE),
    (dict(adv_layout=3), rl.RL_ERR_DTYPE),
    (dict(V=0), rl.RL_ERR_SHAPE),
    (dict(ld=1000), rl.RL_ERR_SHAPE),
    (dict(B=-1), rl.RL_ERR_SHAPE),
    (dict(T=-3), rl.RL_ERR_SHAPE),
    (dict(stats=None), rl.RL_ERR_NULL),
    (dict(ids=None), rl.RL_ERR_NULL),
    (dict(mask=None), rl.RL_ERR_NULL),
    (dict(adv=None), rl.RL_ERR_NULL),
    (dict(logits=None), rl.RL_ERR_NULL),
    (dict(beta=0.1), rl.RL_ERR_NULL),                      # KL without ref_logp
    (dict(workspace=None), rl.RL_ERR_WORKSPACE),
    (dict(ws_bytes=16), rl.RL_ERR_WORKSPACE),
    (dict(eps=float("nan")), rl.RL_ERR_ARG),
    (dict(eps=-0.1), rl.RL_ERR_ARG),
    (dict(grad_scale=float("inf")), rl.RL_ERR_ARG),
    (dict(c_ent=float("nan")), rl.RL_ERR_ARG),
    (dict(V=1001, ld=1001), rl.RL_ERR_ALIGN),             # 2002-byte rows
    (dict(logits=FAKE + 8), rl.RL_ERR_ALIGN),
    (dict(dlogits=FAKE + 0x400002), rl.RL_ERR_ALIGN),
    (dict(dlogits=FAKE + 16), rl.RL_ERR_ALIAS),           # partial overlap
])
def test_loss_argument_errors(lib, over, status):
    assert call_loss(lib, **over) == status


def test_group_advantages_argument_errors(lib):
    f = lib.rl_group_advantages
    assert f(FAKE, 4, 0, 1e-4, 1, FAKE, None) == rl.RL_ERR_SHAPE
    assert f(FAKE, -1, 4, 1e-4, 1, FAKE, None) == rl.RL_ERR_SHAPE
    assert f(FAKE, 4, 1, 1e-4, 1, FAKE, None) == rl.RL_ERR_SHAPE   # G = 1 with ddof = 1
    assert f(FAKE, 4, 4, 1e-4, 2, FAKE, None) == rl.RL_ERR_ARG
    assert f(FAKE, 4, 4, float("nan"), 1, FAKE, None) == rl.RL_ERR_ARG
    assert f(None, 4, 4, 1e-4, 1, FAKE, None) == rl.RL_ERR_NULL
    assert f(None, 0, 4, 1e-4, 1, None, None) == rl.RL_OK         # nothing to do


def test_gae_argument_errors(lib):
    f = lib.rl_gae_reverse_scan
    assert f(FAKE, FAKE, FAKE, -1, 4, 1.0, 0.95, FAKE, None, None) == rl.RL_ERR_SHAPE
    assert f(FAKE, FAKE, FAKE, 4, -1, 1.0, 0.95, FAKE, None, None) == rl.RL_ERR_SHAPE
    assert f(FAKE, FAKE, FAKE, 4, 4, float("nan"), 0.95, FAKE, None, None) == rl.RL_ERR_ARG
    assert f(None, FAKE, FAKE, 4, 4, 1.0, 0.95, FAKE, None, None) == rl.RL_ERR_NULL
    assert f(None, None, None, 0, 4, 1.0, 0.95, None, None, None) == rl.RL_OK


def test_read_status_null(lib):
    assert lib.rl_read_device_status(None, None) == rl.RL_ERR_NULL


def test_binding_raises_without_library(tmp_path):
    with pytest.raises(RuntimeError):
        saved = rl._lib
        rl._lib = None
        try:
            rl.load(str(tmp_path / "missing.so"))
        finally:
            rl._lib = saved


def _desc(**over):
    d = rl.rl_policy_loss_desc_init()
    d.logits, d.dtype, d.B, d.T, d.V, d.ld = FAKE, rl.RL_BF16, 2, 4, 1024, 1024
    d.ids, d.mask, d.adv = FAKE + 0x100000, FAKE + 0x200000, FAKE + 0x300000
    d.dlogits, d.stats_dev, d.workspace = FAKE + 0x400000, FAKE + 0x500000, FAKE + 0x600000
    d.workspace_bytes = rl.rl_policy_loss_workspace_size(8)
    for k, v in over.items():
        setattr(d, k, v)
    return d


def test_desc_defaults(lib):
    d = rl.rl_policy_loss_desc_init()
    assert abs(d.eps - 0.2) < 1e-7 and d.eps_high == -1.0 and d.ddof == 1
    assert d.std_eps == 1e-4 and d.grad_scale == 1.0 and d.agg == rl.RL_AGG_TOKEN_MEAN


@pytest.mark.parametrize("over,status", [
    (dict(agg=9), rl.RL_ERR_DTYPE),
    (dict(adv_layout=5), rl.RL_ERR_DTYPE),
    (dict(agg=rl.RL_AGG_TOKEN_SUM_NORM, agg_norm=0.0), rl.RL_ERR_ARG),
    (dict(agg=rl.RL_AGG_TOKEN_SUM_NORM, agg_norm=float("nan")), rl.RL_ERR_ARG),
    (dict(adv_layout=rl.RL_ADV_GROUP_REWARDS, group_size=3), rl.RL_ERR_SHAPE),  # 3 does not divide B=2
    (dict(adv_layout=rl.RL_ADV_GROUP_REWARDS, group_size=1), rl.RL_ERR_SHAPE),  # G <= ddof
    (dict(adv_layout=rl.RL_ADV_GROUP_REWARDS, group_size=2, ddof=2), rl.RL_ERR_ARG),
    (dict(adv_layout=rl.RL_ADV_GROUP_REWARDS, group_size=2, std_eps=-1.0), rl.RL_ERR_ARG),
    (dict(eps_high=float("inf")), rl.RL_ERR_ARG),
    (dict(stats_dev=None), rl.RL_ERR_NULL),
    # vocabulary shards
    (dict(partials_out=FAKE + 0x700000, shard_partials=FAKE + 0x800000, n_shards=2), rl.RL_ERR_ARG),
    (dict(shard_partials=FAKE + 0x800000, n_shards=0), rl.RL_ERR_ARG),
    (dict(vocab_offset=8, vocab_total=1024), rl.RL_ERR_SHAPE),      # shard runs past the vocabulary
    (dict(vocab_offset=-8, vocab_total=4096), rl.RL_ERR_SHAPE),
    (dict(partials_out=FAKE + 0x700008), rl.RL_ERR_ALIGN),
    # row coefficients for the LM-head backward: merge launches only, 16-byte aligned;
    # a merge launch without columns (V = 0) needs them and the vocabulary size
    (dict(row_coef_out=FAKE + 0x900000), rl.RL_ERR_ARG),
    (dict(shard_partials=FAKE + 0x800000, n_shards=1, row_coef_out=FAKE + 0x900008), rl.RL_ERR_ALIGN),
    (dict(shard_partials=FAKE + 0x800000, n_shards=1, V=0, ld=0), rl.RL_ERR_SHAPE),
    (dict(shard_partials=FAKE + 0x800000, n_shards=1, V=0, ld=0, row_coef_out=FAKE + 0x900000),
     rl.RL_ERR_SHAPE),                                               # no vocab_total
    (dict(shard_partials=FAKE + 0x800000, n_shards=1, V=0, ld=0, vocab_total=1024, logits=None,
          row_coef_out=FAKE + 0x900000, ids=None), rl.RL_ERR_NULL),
])
def test_desc_argument_errors(lib, over, status):
    assert lib.rl_policy_loss_fwd_bwd_ex(ctypes.byref(_desc(**over)), None) == status


def test_desc_null(lib):
    assert lib.rl_policy_loss_fwd_bwd_ex(None, None) == rl.RL_ERR_NULL


def test_fixed_form_rejects_group_rewards_layout(lib):
    assert call_loss(lib, adv_layout=rl.RL_ADV_GROUP_REWARDS) == rl.RL_ERR_DTYPE


def call_lmhead(lib, **over):
    a = dict(hidden=FAKE, ld_h=1024, weight=FAKE + 0x1000000, ld_w=1024, dtype=rl.RL_BF16, R=256,
             D=1024, V=151936,
             ids=FAKE + 0x2000000, logp=FAKE + 0x3000000, ent=None, lse=None, status=None,
             ws=None, ws_bytes=0, stream=None)
    a.update(over)
    return lib.rl_lmhead_logprobs(a["hidden"], a["ld_h"], a["weight"], a["ld_w"], a["dtype"], a["R"], a["D"],
                                  a["V"], a["ids"], a["logp"], a["ent"], a["lse"], a["status"],
                                  a["ws"], a["ws_bytes"], a["stream"])


@pytest.mark.parametrize("over,expect", [
    (dict(R=-1), rl.RL_ERR_SHAPE),
    (dict(dtype=rl.RL_F32), rl.RL_ERR_DTYPE),
    (dict(dtype=7), rl.RL_ERR_DTYPE),
    (dict(D=0), rl.RL_ERR_SHAPE),
    (dict(D=1020, ld_h=1020, ld_w=1020), rl.RL_ERR_SHAPE),    # D not a multiple of 8
    (dict(V=0), rl.RL_ERR_SHAPE),
    (dict(V=(1 << 31) + 1), rl.RL_ERR_SHAPE),
    (dict(ld_h=1000), rl.RL_ERR_SHAPE),                       # stride below D
    (dict(ld_w=512), rl.RL_ERR_SHAPE),
    (dict(hidden=None), rl.RL_ERR_NULL),
    (dict(weight=None), rl.RL_ERR_NULL),
    (dict(ids=None), rl.RL_ERR_NULL),
    (dict(hidden=FAKE + 8), rl.RL_ERR_ALIGN),
    (dict(weight=FAKE + 0x1000002), rl.RL_ERR_ALIGN),
    (dict(ld_h=1028), rl.RL_ERR_ALIGN),                       # row stride not a multiple of 16 B
    (dict(ws=FAKE + 0x4000008, ws_bytes=1 << 20), rl.RL_ERR_ALIGN),
    (dict(R=1 << 31), rl.RL_ERR_SHAPE),
    (dict(R=0), rl.RL_OK),                                    # nothing to launch
])
def test_lmhead_host_errors(lib, over, expect):
    assert call_lmhead(lib, **over) == expect


def test_lmhead_plan_rejects_bad_shapes(lib):
    with pytest.raises(rl.RlLossError):
        rl.rl_lmhead_plan(0, 1024, 1000, 0, 152)
    with pytest.raises(rl.RlLossError):
        rl.rl_lmhead_plan(128, 1024, 0, 0, 152)


@pytest.mark.parametrize("R,V", [(32768, 151936), (65536, 151936), (1024, 151936), (128, 151936),
                                 (16384, 32000), (300, 1000), (40000, 768)])
def test_lmhead_plan_balances_the_sms(lib, R, V):
    """The chosen split keeps the busiest CTA within a few percent of an even
    share of the 128 x 256 tiles (where the tile count allows), and without
    workspace the launch is unsliced."""
    sms = 152
    n_mt, n_nt = -(-R // 128), -(-V // 256)
    ns, grid, grp, need = rl.rl_lmhead_plan(R, 1024, V, 1 << 40, sms)
    assert 1 <= grp <= n_mt
    assert 1 <= ns <= n_nt and grid == min(sms, n_mt * ns)
    if ns > 1:
        assert need >= ns * R * 16 + n_mt * 4
    # busiest CTA under the round-robin deal, in tiles
    load = [0] * grid
    for u in range(n_mt * ns):
        vs = u // n_mt
        load[u % grid] += (vs + 1) * n_nt // ns - vs * n_nt // ns
    ideal = n_mt * n_nt / sms
    if ideal >= 8:
        assert max(load) <= 1.06 * ideal, (ns, max(load), ideal)
    assert rl.rl_lmhead_plan(R, 1024, V, 0, sms)[0] == 1
    assert rl.rl_lmhead_plan(R, 1024, V, 0, sms)[3] == 0


@pytest.mark.parametrize("D,expect", [(1024, 160), (2048, 80), (4096, 40), (200, 640)])
def test_lmhead_plan_groups_row_tiles_to_fit_l2(lib, D, expect):
    """Units are grouped so that the hidden tiles in use at one time (128 rows x D
    bf16 each, D rounded up to 64) stay within a 40 MB share of L2."""
    n_mt = 2000
    grp = rl.rl_lmhead_plan(128 * n_mt, D, 151936, 1 << 40, 152)[2]
    assert grp == min(expect, n_mt)
    assert grp * 128 * (-(-D // 64) * 64) * 2 <= 40 << 20


def test_selftest_wait_timeout_host_errors(lib):
    assert lib.rl_selftest_wait_timeout(1000000, None, None, None) == rl.RL_ERR_NULL
    assert lib.rl_selftest_wait_timeout(10, FAKE, None, None) == rl.RL_ERR_ARG
    assert lib.rl_selftest_wait_timeout(11 * 10**9, FAKE, None, None) == rl.RL_ERR_ARG


# ----------------------------------------------------------------- the LM-head backward entry points
G_DZ, G_W, G_H, G_OUT, G_COEF, G_IDS = (FAKE + k * 0x10000000 for k in range(1, 7))


@pytest.mark.parametrize("over,expect", [
    (dict(dtype=rl.RL_F32), rl.RL_ERR_DTYPE),
    (dict(R=-1), rl.RL_ERR_SHAPE),
    (dict(R=1 << 31), rl.RL_ERR_SHAPE),
    (dict(V=0), rl.RL_ERR_SHAPE),
    (dict(D=1020, ld_h=1020, ld_w=1020), rl.RL_ERR_SHAPE),      # D not a multiple of 8
    (dict(ld_dz=151932), rl.RL_ERR_SHAPE),                      # below V
    (dict(ld_dz=151937, V=151937), rl.RL_ERR_SHAPE),            # not a multiple of 8 elements
    (dict(coef=None), rl.RL_ERR_NULL),
    (dict(ids=None), rl.RL_ERR_NULL),
    (dict(out=None), rl.RL_ERR_NULL),
    (dict(coef=G_COEF + 8), rl.RL_ERR_ALIGN),
    (dict(out=G_OUT + 2), rl.RL_ERR_ALIGN),
    (dict(R=0, coef=None, out=None), rl.RL_OK),                  # nothing to launch
])
def test_lmhead_dlogits_host_errors(lib, over, expect):
    a = dict(h=G_H, ld_h=1024, w=G_W, ld_w=1024, dtype=rl.RL_BF16, R=256, D=1024, V=151936,
             ids=G_IDS, coef=G_COEF, out=G_OUT, ld_dz=151936)
    a.update(over)
    assert lib.rl_lmhead_dlogits(a["h"], a["ld_h"], a["w"], a["ld_w"], a["dtype"], a["R"], a["D"],
                                 a["V"], a["ids"], a["coef"], a["out"], a["ld_dz"], None,
                                 None) == expect


@pytest.mark.parametrize("over,expect", [
    (dict(dtype=7), rl.RL_ERR_DTYPE),
    (dict(D=4), rl.RL_ERR_SHAPE),
    (dict(ld_dh=512), rl.RL_ERR_SHAPE),
    (dict(dz=None), rl.RL_ERR_NULL),
    (dict(out=None), rl.RL_ERR_NULL),
    (dict(w=G_W + 4), rl.RL_ERR_ALIGN),
    (dict(R=0, dz=None), rl.RL_OK),
])
def test_lmhead_dhidden_host_errors(lib, over, expect):
    a = dict(dz=G_DZ, ld_dz=151936, w=G_W, ld_w=1024, dtype=rl.RL_BF16, R=256, D=1024, V=151936,
             out=G_OUT, ld_dh=1024)
    a.update(over)
    assert lib.rl_lmhead_dhidden(a["dz"], a["ld_dz"], a["w"], a["ld_w"], a["dtype"], a["R"], a["D"],
                                 a["V"], a["out"], a["ld_dh"], None, None) == expect


@pytest.mark.parametrize("over,expect", [
    (dict(dtype=rl.RL_F32), rl.RL_ERR_DTYPE),
    (dict(ld_dw=1022), rl.RL_ERR_SHAPE),                          # below D
    (dict(ld_dw=1030), rl.RL_ERR_SHAPE),                          # not a multiple of 4 floats
    (dict(out=None), rl.RL_ERR_NULL),
    (dict(out=G_OUT + 4), rl.RL_ERR_ALIGN),
    (dict(dz=None), rl.RL_ERR_NULL),
    (dict(h=G_H + 2), rl.RL_ERR_ALIGN),
    (dict(R=0, dz=None, h=None, acc=1), rl.RL_OK),               # adds nothing
])
def test_lmhead_dweight_host_errors(lib, over, expect):
    a = dict(dz=G_DZ, ld_dz=151936, h=G_H, ld_h=1024, dtype=rl.RL_BF16, R=256, D=1024, V=151936,
             out=G_OUT, ld_dw=1024, acc=0)
    a.update(over)
    assert lib.rl_lmhead_dweight(a["dz"], a["ld_dz"], a["h"], a["ld_h"], a["dtype"], a["R"], a["D"],
                                 a["V"], a["out"], a["ld_dw"], a["acc"], None, None) == expect


def test_lmhead_row_partials_host_errors(lib):
    f = lib.rl_lmhead_row_partials
    args = [FAKE, 1024, FAKE + 0x1000000, 1024, rl.RL_BF16, 256, 1024, 151936, FAKE + 0x2000000]
    assert f(*args, None, None, None, 0, None) == rl.RL_ERR_NULL               # no output
    assert f(*args, FAKE + 0x3000008, None, None, 0, None) == rl.RL_ERR_ALIGN  # 16-byte records
    bad = list(args)
    bad[4] = rl.RL_F32
    assert f(*bad, FAKE + 0x3000000, None, None, 0, None) == rl.RL_ERR_DTYPE
