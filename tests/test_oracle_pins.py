"""Pins for the CPU oracle: checks against things other than the oracle itself.

Each test pins one part of the oracle to a library routine, a closed form, an
invariant of the mathematics, a brute-force computation or a hand-worked table
(tests/golden/).  A plausible slip in the oracle (a dropped term, a wrong
sign or index, a transposed operand) fails at least one of them.
"""
import math
import os

import numpy as np
import pytest
import scipy.special
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ----------------------------------------------------------------------------- formats
def test_decode_bf16_all_patterns_match_torch():
    bits = np.arange(1 << 16, dtype=np.uint16)
    ours = oracle.decode(bits, "bf16")
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).double().numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])


def test_decode_f16_all_patterns_match_numpy():
    bits = np.arange(1 << 16, dtype=np.uint16)
    ours = oracle.decode(bits, "f16")
    ref = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])


def _float32_values(n, seed):
    rng = np.random.default_rng(seed)
    bits = rng.integers(0, 1 << 32, size=n, dtype=np.uint64).astype(np.uint32)
    x = bits.view(np.float32)
    x = x[np.isfinite(x)]
    extra = np.array([0.0, -0.0, 1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, 65504.0, 65520.0,
                      3.3895314e38, 3.40282347e38, 1e-45, 2 ** -126, 2 ** -133, 2 ** -24,
                      2 ** -25, 3 * 2 ** -26, 6.1e-5], np.float32)
    return np.concatenate([x, extra, -extra])


def test_encode_bf16_matches_torch_on_float32_inputs():
    # torch rounds binary32 -> bfloat16 to nearest even; every binary32 value is a double,
    # so on these inputs the oracle's single rounding must agree bit for bit.
    x = _float32_values(200_000, 1)
    ours = oracle.encode(x.astype(np.float64), "bf16")
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)


def test_encode_bf16_rounds_once_from_double():
    # 1 + 2^-8 + 2^-30 lies above the midpoint between 1 and 1 + 2^-7: one rounding gives
    # 1 + 2^-7 (0x3F81); rounding through binary32 first would tie and give 1.0.
    got = oracle.encode(np.array([1 + 2 ** -8 + 2 ** -30, 1 + 2 ** -8, 1 + 3 * 2 ** -8]), "bf16")
    assert list(got) == [0x3F81, 0x3F80, 0x3F82]


def test_encode_f16_matches_numpy():
    rng = np.random.default_rng(2)
    x = np.concatenate([rng.normal(0, 1, 100_000) * 10.0 ** rng.integers(-9, 6, 100_000),
                        [65504.0, 65519.99, 65520.0, 1e6, 2 ** -24, 2 ** -25, 1.5 * 2 ** -25,
                         2 ** -14, 1 + 2 ** -11 + 2 ** -40, 0.0, -0.0]])
    ours = oracle.encode(x, "f16")
    ref = x.astype(np.float16).view(np.uint16)
    assert np.array_equal(ours, ref)


def test_encode_f32_matches_numpy():
    x = np.random.default_rng(3).normal(0, 1, 10_000) * 1e-30
    assert np.array_equal(oracle.encode(x, "f32"), x.astype(np.float32))


def test_ulp_matches_numpy_spacing():
    x = np.array([1.0, 3.0, 1e-3, 100.0, 6e-5])
    assert np.array_equal(oracle.ulp(x, "f32"), np.spacing(x.astype(np.float32)).astype(np.float64))
    assert np.array_equal(oracle.ulp(x, "f16"), np.spacing(x.astype(np.float16)).astype(np.float64))


# ----------------------------------------------------------------------------- row statistics
def _stats64(z, ids, mask=None):
    z = np.ascontiguousarray(z, np.float64)
    m = np.ones(z.shape[0], np.uint8) if mask is None else mask
    return oracle.row_stats(z, "f64", z.shape[1], ids, m, threads=1)


def test_row_stats_match_scipy():
    rng = np.random.default_rng(4)
    z = rng.normal(0, 3, (7, 513))
    ids = rng.integers(0, 513, 7)
    lse, logp, H = _stats64(z, ids)
    ref_lse = scipy.special.logsumexp(z, axis=1)
    ref_lsm = scipy.special.log_softmax(z, axis=1)
    ref_H = scipy.stats.entropy(scipy.special.softmax(z, axis=1), axis=1)
    np.testing.assert_allclose(lse, ref_lse, rtol=1e-13)
    np.testing.assert_allclose(logp, ref_lsm[np.arange(7), ids], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(H, ref_H, rtol=1e-12)


def test_uniform_logits_closed_form():
    for V in (1, 2, 1024, 151936):
        z = np.full((1, V), 1.7)
        lse, logp, H = _stats64(z, np.array([V - 1]))
        assert abs(logp[0] + math.log(V)) < 1e-12
        assert abs(H[0] - math.log(V)) < 1e-10 * max(1.0, math.log(V))
        assert abs(lse[0] - (1.7 + math.log(V))) < 1e-12


def test_one_hot_logits_closed_form():
    V, k = 1000, 17
    z = np.zeros((2, V))
    z[:, k] = 100.0
    lse, logp, H = _stats64(z, np.array([k, 3]))
    q = math.exp(-100.0)                         # p_v / p_k for v != k
    pk = 1.0 / (1.0 + (V - 1) * q)
    assert abs(logp[0] - math.log(pk)) < 1e-15
    assert abs(logp[1] - (-100.0 + math.log(pk))) < 1e-12
    H_exact = -(pk * math.log(pk) + (V - 1) * (q * pk) * math.log(q * pk))
    assert abs(H[0] - H_exact) < 1e-30


def test_two_logits_binary_closed_form():
    a, b = 0.3, -1.9
    lse, logp, H = _stats64(np.array([[a, b]]), np.array([0]))
    p0 = 1.0 / (1.0 + math.exp(b - a))
    assert abs(logp[0] - math.log(p0)) < 1e-15
    assert abs(H[0] - (-(p0 * math.log(p0) + (1 - p0) * math.log(1 - p0)))) < 1e-15


def test_shift_invariance():
    rng = np.random.default_rng(5)
    z = rng.normal(0, 2, (3, 300))
    ids = np.array([0, 150, 299])
    lse0, logp0, H0 = _stats64(z, ids)
    lse1, logp1, H1 = _stats64(z + 37.25, ids)
    np.testing.assert_allclose(logp1, logp0, atol=1e-12)
    np.testing.assert_allclose(H1, H0, atol=1e-12)
    np.testing.assert_allclose(lse1, lse0 + 37.25, atol=1e-12)


def test_large_vocab_lse_aggregate():
    # For z ~ N(0, sd) iid, lse = ln V + ln mean(e^z) -> ln V + sd^2/2 as V grows.
    rng = np.random.default_rng(6)
    V, sd = 151936, 1.0
    z = rng.normal(0, sd, (4, V))
    lse, _, _ = _stats64(z, np.zeros(4, np.int64))
    assert np.all(np.abs(lse - (math.log(V) + sd * sd / 2)) < 0.02)


def test_masked_rows_and_bad_ids():
    z = np.random.default_rng(7).normal(0, 1, (3, 10))
    lse, logp, H = oracle.row_stats(z, "f64", 10, np.array([1, 10, -1]),
                                    np.array([0, 1, 1], np.uint8), threads=1)
    assert lse[0] == 0 and logp[0] == 0 and H[0] == 0
    assert np.isnan(logp[1]) and np.isnan(logp[2])


def test_low_precision_rows_decode_exactly():
    # A bf16 row and the same row widened to f64 must give identical statistics.
    x = torch.randn(2, 777, generator=torch.Generator().manual_seed(8)).mul(3).to(torch.bfloat16)
    st = x.view(torch.int16).numpy().view(np.uint16)
    ids = np.array([5, 700])
    a = oracle.row_stats(st, "bf16", 777, ids, np.ones(2, np.uint8), threads=1)
    b = _stats64(x.double().numpy(), ids)
    for u, v in zip(a, b):
        assert np.array_equal(u, v)


# ----------------------------------------------------------------------------- advantages
def test_group_advantages_vs_numpy_std():
    rng = np.random.default_rng(9)
    R = rng.random(8 * 6)
    for ddof in (0, 1):
        A = oracle.group_advantages(R, 6, 1e-4, ddof)
        g = R.reshape(8, 6)
        ref = (g - g.mean(1, keepdims=True)) / (g.std(1, ddof=ddof, keepdims=True) + 1e-4)
        np.testing.assert_allclose(A, ref.reshape(-1), rtol=1e-12, atol=1e-13)
        assert np.all(np.abs(A.reshape(8, 6).sum(1)) < 1e-12)


def test_group_advantages_equal_rewards_are_zero():
    R = np.array([1, 1, 1, 1, 0, 0, 0, 0, 1, 0, 1, 1], np.float64)
    A = oracle.group_advantages(R, 4)
    assert np.all(A[:8] == 0.0)
    assert np.all(A[8:] != 0.0)


def test_group_advantages_pair_closed_form():
    # G = 2, ddof = 1: std = |dR| / sqrt(2), so A = +/- (|dR|/2) / (|dR|/sqrt(2) + eps).
    R = np.array([0.25, 1.0])
    A = oracle.group_advantages(R, 2)
    d = 0.75
    expect = (d / 2) / (d / math.sqrt(2) + 1e-4)
    assert abs(A[1] - expect) < 1e-15 and abs(A[0] + expect) < 1e-15


def _gae_inputs(seed, B=5, T=40):
    rng = np.random.default_rng(seed)
    r = rng.normal(0, 1, (B, T))
    v = rng.normal(0, 0.5, (B, T))
    L = np.array([T, 1, 0, T // 2, T - 3])[:B]
    return r, v, L


def test_gae_lambda_zero_is_td_error():
    r, v, L = _gae_inputs(10)
    A, ret = oracle.gae(r, v, L, 0.9, 0.0)
    for b in range(r.shape[0]):
        for t in range(L[b]):
            vn = v[b, t + 1] if t + 1 < L[b] else 0.0
            assert abs(A[b, t] - (r[b, t] + 0.9 * vn - v[b, t])) < 1e-12
        assert np.all(A[b, L[b]:] == 0) and np.all(ret[b, L[b]:] == 0)


def test_gae_gamma_lambda_one_is_reward_to_go():
    r, v, L = _gae_inputs(11)
    A, ret = oracle.gae(r, v, L, 1.0, 1.0)
    for b in range(r.shape[0]):
        for t in range(L[b]):
            assert abs(A[b, t] - (r[b, t:L[b]].sum() - v[b, t])) < 1e-10
            assert abs(ret[b, t] - r[b, t:L[b]].sum()) < 1e-10


def test_gae_brute_force_sum():
    r, v, L = _gae_inputs(12)
    gamma, lam = 0.99, 0.95
    A, ret = oracle.gae(r, v, L, gamma, lam)
    for b in range(r.shape[0]):
        Lb = L[b]
        delta = [r[b, k] + gamma * (v[b, k + 1] if k + 1 < Lb else 0.0) - v[b, k] for k in range(Lb)]
        for t in range(Lb):
            bf = sum((gamma * lam) ** (k - t) * delta[k] for k in range(t, Lb))
            assert abs(A[b, t] - bf) < 1e-10
            assert abs(ret[b, t] - (bf + v[b, t])) < 1e-10


def test_gae_constant_delta_geometric():
    # r_t = d + V_t - gamma V_{t+1} makes delta_t = d everywhere.
    T, gamma, lam, d = 30, 0.97, 0.9, 0.3
    v = np.linspace(-1, 1, T)[None, :]
    vn = np.append(v[0, 1:], 0.0)
    r = (d + v[0] - gamma * vn)[None, :]
    A, _ = oracle.gae(r, v, np.array([T]), gamma, lam)
    c = gamma * lam
    for t in range(T):
        n = T - t
        assert abs(A[0, t] - d * (1 - c ** n) / (1 - c)) < 1e-12


# ----------------------------------------------------------------------------- objective
def _golden_clip(name="clip_cases.txt"):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append([float(x) for x in line.split()])
    return np.array(rows)


def test_surrogate_hand_table():
    tab = _golden_clip()
    A, r, pg, dpg, clipped = tab.T
    got_pg, got_dpg, got_clipped = oracle.surrogate(r, A, 0.2)
    np.testing.assert_allclose(got_pg, pg, atol=1e-15)
    np.testing.assert_allclose(got_dpg, dpg, atol=1e-15)
    assert np.array_equal(got_clipped, clipped.astype(bool))


def test_surrogate_clip_higher_hand_table():
    A, r, pg, dpg, clipped = _golden_clip("clip_higher_cases.txt").T
    got_pg, got_dpg, got_clipped = oracle.surrogate(r, A, 0.2, 0.28)
    np.testing.assert_allclose(got_pg, pg, atol=1e-15)
    np.testing.assert_allclose(got_dpg, dpg, atol=1e-15)
    assert np.array_equal(got_clipped, clipped.astype(bool))


def test_surrogate_brute_force_derivative():
    # Away from the clip boundaries, dpg equals the numerical derivative of
    # pg(exp(l - l_old)) in l: brute force over a grid of A and r.
    eps, h = 0.2, 1e-7
    for A in (-2.0, -0.3, 0.0, 0.7, 1.5):
        for r in np.linspace(0.5, 1.5, 41):
            if min(abs(r - 0.8), abs(r - 1.2)) < 1e-3:
                continue
            l = math.log(r)
            pg_p = oracle.surrogate(math.exp(l + h), A, eps)[0]
            pg_m = oracle.surrogate(math.exp(l - h), A, eps)[0]
            fd = (pg_p - pg_m) / (2 * h)
            assert abs(oracle.surrogate(r, A, eps)[1] - fd) < 1e-6


def test_one_sided_derivatives_at_the_clip_kink():
    # With the ratio exactly on a clip boundary the surrogate has a kink: the
    # derivative of J in logp from one side is the unclipped branch (r A +
    # KL term), from the other the clipped one (KL term only).  Which side is
    # which depends on the sign of A.  One-sided differences of the oracle's
    # own J pin g_unclipped and g_clipped; away from the kink g is one of them.
    eps, beta, h = 0.2, 0.3, 1e-7
    lo_ref = -1.3
    for A, r_b in ((0.9, 1 + eps), (-0.7, 1 - eps), (1.4, 1 - eps), (-2.0, 1 + eps)):
        lo = -2.0
        l0 = lo + math.log(r_b)
        m = np.ones(1, np.uint8)

        def J(l):
            return oracle.token_objective(np.array([l]), np.zeros(1), m, np.array([A]),
                                          np.array([lo]), np.array([lo_ref]), eps, beta, 0.0)["J"][0]

        o = oracle.token_objective(np.array([l0]), np.zeros(1), m, np.array([A]), np.array([lo]),
                                   np.array([lo_ref]), eps, beta, 0.0)
        right = (J(l0 + h) - J(l0)) / h
        left = (J(l0) - J(l0 - h)) / h
        # r grows with logp.  The clip binds above 1 + eps when A > 0 and below
        # 1 - eps when A < 0; at the other boundary there is no kink.
        if A > 0 and r_b > 1:
            free_side, clipped_side = left, right
        elif A < 0 and r_b < 1:
            free_side, clipped_side = right, left
        else:
            free_side, clipped_side = left, None
            assert abs(right - o["g_unclipped"][0]) < 1e-5, (A, r_b)
        assert abs(free_side - o["g_unclipped"][0]) < 1e-5, (A, r_b)
        if clipped_side is not None:
            assert abs(clipped_side - o["g_clipped"][0]) < 1e-5, (A, r_b)
        # at the boundary itself the gradient flows (inclusive clip): g is the unclipped branch
        assert o["g"][0] == o["g_unclipped"][0]
    z, ids, mask, adv, n_old, n_ref = _problem(29, R=40)
    _, logp, H = oracle.row_stats(z, "f64", z.shape[1], ids, mask, threads=1)
    o = oracle.token_objective(logp, H, mask, 3 * adv, logp + 3 * n_old, logp + n_ref, 0.05, 0.2, 0.0)
    assert o["clipped"].any() and (~o["clipped"] & (mask != 0)).any()
    assert np.array_equal(o["g"], np.where(o["clipped"], o["g_clipped"], o["g_unclipped"]))


def test_kl_k3_zero_at_reference_and_quadratic_small():
    logp = np.array([-3.0, -1.0, -0.5])
    m = np.ones(3, np.uint8)
    o = oracle.token_objective(logp, np.zeros(3), m, np.zeros(3), None, logp.copy(), 0.2, 1.0, 0.0)
    assert np.all(o["kl"] == 0) and np.all(o["g"] == 0)
    d = 1e-3
    o = oracle.token_objective(logp, np.zeros(3), m, np.zeros(3), None, logp + d, 0.2, 1.0, 0.0)
    np.testing.assert_allclose(o["kl"], d * d / 2 + d ** 3 / 6, rtol=1e-6)


def _problem(seed, R=12, V=9, T=4, **kw):
    rng = np.random.default_rng(seed)
    z = rng.normal(0, 1.5, (R, V))
    ids = rng.integers(0, V, R)
    mask = (rng.random(R) < 0.75).astype(np.uint8)
    mask[0] = 1
    adv = rng.normal(0, 1, R)
    noise_old = rng.normal(0, 0.1, R)
    noise_ref = rng.normal(0, 0.3, R)
    return z, ids, mask, adv, noise_old, noise_ref


def test_on_policy_no_kl_loss_identity():
    # logp == logp_old and beta = 0: r = 1 (never clipped), so
    # loss = -mean(A) - c_ent mean(H) over the valid tokens.
    z, ids, mask, adv, _, _ = _problem(13)
    V = z.shape[1]
    _, logp, H = oracle.row_stats(z, "f64", V, ids, mask, threads=1)
    out = oracle.policy_loss(z, "f64", V, ids, mask, adv, logp_old=logp, ref_logp=None,
                             eps=0.2, beta=0.0, c_ent=0.05, grad_rows=False)
    mb = mask.astype(bool)
    assert abs(out["loss"] - (-adv[mb].mean() - 0.05 * H[mb].mean())) < 1e-12
    assert out["n_clipped"] == 0


def test_loss_linear_and_odd_in_advantage():
    z, ids, mask, adv, _, _ = _problem(14)
    V = z.shape[1]
    _, logp, _ = oracle.row_stats(z, "f64", V, ids, mask, threads=1)
    f = lambda a: oracle.policy_loss(z, "f64", V, ids, mask, a, logp_old=logp, eps=0.2,
                                     grad_rows=False)["loss"]
    assert abs(f(2.5 * adv) - 2.5 * f(adv)) < 1e-12
    assert abs(f(-adv) + f(adv)) < 1e-12


def test_zero_valid_tokens():
    z, ids, _, adv, _, _ = _problem(15)
    mask = np.zeros(z.shape[0], np.uint8)
    out = oracle.policy_loss(z, "f64", z.shape[1], ids, mask, adv, eps=0.2, beta=0.1, c_ent=0.1,
                             ref_logp=np.zeros(z.shape[0]), out_dtype="f64")
    assert out["loss"] == 0 and out["n_tokens"] == 0
    assert np.all(out["dlogits"] == 0)


# ----------------------------------------------------------------------------- gradient
@pytest.mark.parametrize("V", [2, 3, 8, 17])
def test_dlogits_central_differences(V):
    z, ids, mask, adv, n_old, n_ref = _problem(20 + V, R=10, V=V)
    _, logp0, _ = oracle.row_stats(z, "f64", V, ids, mask, threads=1)
    logp_old = logp0 + n_old
    ref = logp0 + n_ref
    # keep every ratio well away from the clip boundaries, where pg is not differentiable
    r = np.exp(logp0 - logp_old)
    for i in range(len(r)):
        if min(abs(r[i] - 0.8), abs(r[i] - 1.2)) < 1e-3:
            logp_old[i] += 0.01
    # force a clipped token on each side
    logp_old[0] = logp0[0] - 0.5
    adv[0] = abs(adv[0]) + 0.1
    kw = dict(eps=0.2, beta=0.07, c_ent=0.03, logp_old=logp_old, ref_logp=ref)
    out = oracle.policy_loss(z, "f64", V, ids, mask, adv, grad_scale=1.0, out_dtype="f64", **kw)
    assert out["n_clipped"] >= 1
    h = 1e-6
    fd = np.zeros_like(z)
    for i in range(z.shape[0]):
        for v in range(V):
            zp, zm = z.copy(), z.copy()
            zp[i, v] += h
            zm[i, v] -= h
            lp = oracle.policy_loss(zp, "f64", V, ids, mask, adv, grad_rows=False, **kw)["loss"]
            lm = oracle.policy_loss(zm, "f64", V, ids, mask, adv, grad_rows=False, **kw)["loss"]
            fd[i, v] = (lp - lm) / (2 * h)
    np.testing.assert_allclose(out["dlogits"], fd, rtol=1e-6, atol=1e-9)


def test_dlogits_rows_sum_to_zero_and_masked_rows_zero():
    z, ids, mask, adv, n_old, n_ref = _problem(30, R=16, V=200)
    _, logp0, _ = oracle.row_stats(z, "f64", 200, ids, mask, threads=1)
    out = oracle.policy_loss(z, "f64", 200, ids, mask, adv, logp_old=logp0 + n_old,
                             ref_logp=logp0 + n_ref, eps=0.2, beta=0.04, c_ent=0.01,
                             grad_scale=16.0, out_dtype="f64")
    d = out["dlogits"]
    assert np.all(np.abs(d.sum(1)) < 1e-13)
    assert np.all(d[mask == 0] == 0)
    assert np.any(d[mask == 1] != 0)


def test_sft_corner_is_softmax_minus_onehot():
    # A = 1, on-policy, beta = c_ent = 0, grad_scale = N: dz = softmax(z) - onehot(y),
    # the textbook cross-entropy gradient (torch.softmax in float64 as the reference).
    z, ids, _, _, _, _ = _problem(31, R=6, V=50)
    mask = np.ones(6, np.uint8)
    out = oracle.policy_loss(z, "f64", 50, ids, mask, np.ones(6), eps=0.2,
                             grad_scale=6.0, out_dtype="f64")
    ref = torch.softmax(torch.from_numpy(z), dim=1).numpy()
    ref[np.arange(6), ids] -= 1.0
    np.testing.assert_allclose(out["dlogits"], ref, atol=1e-15)
    # and the loss is the mean cross-entropy minus... nothing: -mean(A r) = -1
    assert abs(out["loss"] + 1.0) < 1e-15


def test_dlogits_rounding_to_bf16_is_single_rounding():
    z, ids, mask, adv, _, _ = _problem(32, R=8, V=64)
    kw = dict(eps=0.2, c_ent=0.02, grad_scale=8.0)
    d64 = oracle.policy_loss(z, "f64", 64, ids, mask, adv, out_dtype="f64", **kw)["dlogits"]
    d16 = oracle.policy_loss(z, "f64", 64, ids, mask, adv, out_dtype="bf16", **kw)["dlogits"]
    assert np.array_equal(d16, oracle.encode(d64, "bf16"))


# ----------------------------------------------------------------------------- aggregations
def _seq_problem(seed, B=6, T=7, V=11, lengths=None):
    rng = np.random.default_rng(seed)
    z = rng.normal(0, 1.5, (B * T, V))
    ids = rng.integers(0, V, B * T)
    L = rng.integers(0, T + 1, B) if lengths is None else np.asarray(lengths)
    mask = (np.arange(T)[None, :] < L[:, None]).astype(np.uint8).reshape(-1)
    adv = np.repeat(rng.normal(0, 1, B), T)
    _, logp0, _ = oracle.row_stats(z, "f64", V, ids, mask, threads=1)
    lo = logp0 + rng.normal(0, 0.1, B * T)
    rf = logp0 + rng.normal(0, 0.2, B * T)
    return z, ids, mask, adv, lo, rf, L


def _loss(z, ids, mask, adv, lo, rf, T, agg, agg_norm=None, **kw):
    return oracle.policy_loss(z, "f64", z.shape[1], ids, mask, adv, logp_old=lo, ref_logp=rf,
                              eps=0.2, beta=0.05, c_ent=0.02, agg=agg, T=T, agg_norm=agg_norm,
                              grad_rows=False, **kw)["loss"]


def test_token_sum_over_N_is_token_mean():
    z, ids, mask, adv, lo, rf, L = _seq_problem(40)
    N = int(mask.sum())
    a = _loss(z, ids, mask, adv, lo, rf, 7, "token_mean")
    b = _loss(z, ids, mask, adv, lo, rf, 7, "token_sum_norm", agg_norm=N)
    assert abs(a - b) < 1e-13


def test_sequence_means_with_equal_lengths_reduce_to_token_mean():
    z, ids, mask, adv, lo, rf, L = _seq_problem(41, lengths=[5, 5, 5, 5, 5, 5])
    a = _loss(z, ids, mask, adv, lo, rf, 7, "token_mean")
    b = _loss(z, ids, mask, adv, lo, rf, 7, "seq_mean_token_mean")
    c = _loss(z, ids, mask, adv, lo, rf, 7, "seq_mean_token_sum")
    assert abs(a - b) < 1e-13
    assert abs(c - 5 * a) < 1e-12


def test_sequence_mean_ignores_empty_sequences_and_weights_each_sequence_equally():
    # one sequence alone gives its own token mean; adding an empty sequence changes nothing;
    # two sequences give the plain average of their two token means
    z, ids, mask, adv, lo, rf, L = _seq_problem(42, B=3, lengths=[3, 0, 6])
    only0 = mask.copy().reshape(3, 7)
    only0[2] = 0
    only2 = mask.copy().reshape(3, 7)
    only2[0] = 0
    m0 = _loss(z, ids, only0.reshape(-1), adv, lo, rf, 7, "token_mean")
    m2 = _loss(z, ids, only2.reshape(-1), adv, lo, rf, 7, "token_mean")
    both = _loss(z, ids, mask, adv, lo, rf, 7, "seq_mean_token_mean")
    assert abs(both - (m0 + m2) / 2) < 1e-13
    assert abs(_loss(z, ids, only0.reshape(-1), adv, lo, rf, 7, "seq_mean_token_mean") - m0) < 1e-13


@pytest.mark.parametrize("agg", oracle.AGGREGATIONS)
def test_dlogits_central_differences_every_aggregation(agg):
    z, ids, mask, adv, lo, rf, L = _seq_problem(43, B=4, T=3, V=5, lengths=[3, 1, 0, 2])
    kw = dict(eps=0.2, eps_high=0.3, beta=0.07, c_ent=0.03, logp_old=lo, ref_logp=rf, agg=agg,
              T=3, agg_norm=9.0)
    out = oracle.policy_loss(z, "f64", 5, ids, mask, adv, grad_scale=1.0, out_dtype="f64", **kw)
    h = 1e-6
    fd = np.zeros_like(z)
    for i in range(z.shape[0]):
        for v in range(5):
            zp, zm = z.copy(), z.copy()
            zp[i, v] += h
            zm[i, v] -= h
            fd[i, v] = (oracle.policy_loss(zp, "f64", 5, ids, mask, adv, grad_rows=False, **kw)["loss"]
                        - oracle.policy_loss(zm, "f64", 5, ids, mask, adv, grad_rows=False, **kw)["loss"]) / (2 * h)
    np.testing.assert_allclose(out["dlogits"], fd, rtol=1e-6, atol=1e-9)


# ----------------------------------------------------------------------------- critic
def test_value_loss_hand_table():
    v, vo, ret, L, dv = _golden_clip("value_clip_cases.txt").T
    n = v.size
    o = oracle.value_loss(v, vo, ret, np.ones(n), clip_eps=0.2, grad_scale=n)
    assert abs(o["loss"] - L.mean()) < 1e-15
    np.testing.assert_allclose(o["dvalues"], dv, atol=1e-15)
    assert o["n_clipped"] == 1


def test_value_loss_unclipped_is_half_mse():
    rng = np.random.default_rng(50)
    v, ret = rng.normal(0, 1, 300), rng.normal(0, 1, 300)
    m = (rng.random(300) < 0.7).astype(np.uint8)
    o = oracle.value_loss(v, None, ret, m)
    assert abs(o["loss"] - 0.5 * np.mean((v - ret)[m == 1] ** 2)) < 1e-14
    # a clip range wider than every step changes nothing
    o2 = oracle.value_loss(v, v + 0.01, ret, m, clip_eps=10.0)
    assert abs(o2["loss"] - o["loss"]) < 1e-15 and o2["n_clipped"] == 0


def test_value_loss_central_differences():
    rng = np.random.default_rng(51)
    v, vo, ret = rng.normal(0, 1, 40), rng.normal(0, 1, 40), rng.normal(0, 1, 40)
    m = (rng.random(40) < 0.8).astype(np.uint8)
    keep = (np.abs(np.abs(v - vo) - 0.3) > 1e-3)  # away from the clip kinks
    v, vo, ret, m = v[keep], vo[keep], ret[keep], m[keep]
    o = oracle.value_loss(v, vo, ret, m, clip_eps=0.3)
    h = 1e-6
    for i in range(v.size):
        vp, vm = v.copy(), v.copy()
        vp[i] += h
        vm[i] -= h
        fd = (oracle.value_loss(vp, vo, ret, m, 0.3)["loss"] - oracle.value_loss(vm, vo, ret, m, 0.3)["loss"]) / (2 * h)
        assert abs(fd - o["dvalues"][i]) < 1e-7


# ----------------------------------------------------------------------------- whitening
def test_masked_whiten_matches_numpy_and_normalises():
    rng = np.random.default_rng(60)
    x = rng.normal(3.0, 2.5, 1000)
    m = (rng.random(1000) < 0.6).astype(np.uint8)
    w = oracle.masked_whiten(x, m, eps=0.0)
    sel = x[m == 1]
    np.testing.assert_allclose(w[m == 1], (sel - sel.mean()) / sel.std(ddof=1), rtol=1e-12)
    assert np.all(w[m == 0] == 0)
    assert abs(w[m == 1].mean()) < 1e-12 and abs(w[m == 1].std(ddof=1) - 1.0) < 1e-12
    w2 = oracle.masked_whiten(x, m, eps=0.0, shift_mean=False)
    np.testing.assert_allclose(w2[m == 1], sel / sel.std(ddof=1), rtol=1e-12)


def test_masked_whiten_degenerate():
    assert np.all(oracle.masked_whiten([1.0, 2.0], [0, 0]) == 0)
    one = oracle.masked_whiten([5.0, 7.0], [0, 1], eps=4.0)
    assert one[1] == 0.0 and one[0] == 0.0          # single token: x - mu = 0
    assert abs(oracle.masked_whiten([5.0], [1], eps=4.0, shift_mean=False)[0] - 2.5) < 1e-15


def test_global_counts_split_batch_shares_sum_to_the_whole():
    # a batch split by sequences over two "ranks": with the whole batch's counts,
    # the two shares of every mean add up to the single-batch value
    z, ids, mask, adv, lo, rf, L = _seq_problem(70, B=6, T=7, lengths=[7, 3, 0, 5, 1, 6])
    V = z.shape[1]
    lse, logp, ent = oracle.row_stats(z, "f64", V, ids, mask, threads=1)
    Bp = int((L > 0).sum())
    gc = (int(mask.sum()), Bp)
    for agg in oracle.AGGREGATIONS:
        kw = dict(eps=0.2, beta=0.05, c_ent=0.02, agg=agg, T=7, agg_norm=30.0)
        whole = oracle.loss_from_stats(logp, ent, mask, adv, lo, rf, **kw)
        parts = [oracle.loss_from_stats(logp[sl], ent[sl], mask[sl], adv[sl], lo[sl], rf[sl],
                                        global_counts=gc, **kw)
                 for sl in (slice(0, 21), slice(21, 42))]
        for k in ("loss", "pg_term", "kl_term", "ent_term", "clip_frac"):
            assert abs(sum(p[k] for p in parts) - whole[k]) < 1e-13, (agg, k)
        assert np.allclose(np.concatenate([p["weights"] for p in parts]), whole["weights"])


# ----------------------------------------------------------------------------- LM head
def test_lmhead_row_stats_match_torch_fp64():
    g = torch.Generator().manual_seed(90)
    h = torch.randn(9, 192, generator=g).to(torch.bfloat16)
    w = (torch.randn(333, 192, generator=g) * 0.2).to(torch.bfloat16)
    ids = torch.randint(0, 333, (9,), generator=g)
    st = lambda t: t.view(torch.int16).numpy().view(np.uint16)
    lse, logp, H = oracle.lmhead_row_stats(st(h), st(w), ids.numpy(), "bf16", threads=1)
    z = h.double() @ w.double().T
    ref_lsm = torch.log_softmax(z, dim=1)
    np.testing.assert_allclose(lse, torch.logsumexp(z, 1).numpy(), rtol=1e-13)
    np.testing.assert_allclose(logp, ref_lsm[torch.arange(9), ids].numpy(), atol=1e-12)
    np.testing.assert_allclose(H, -(ref_lsm.exp() * ref_lsm).sum(1).numpy(), rtol=1e-12)


def test_lmhead_one_hot_hidden_selects_weight_columns():
    """A one-hot hidden state e_k makes the logits the k-th column of W
    (z_v = W[v, k]), so the statistics reduce to scipy's logsumexp over that
    column; a transposed or mis-indexed product fails this."""
    from scipy.special import logsumexp
    g = torch.Generator().manual_seed(91)
    V, D = 50, 24
    w = (torch.randn(V, D, generator=g) * 3).to(torch.bfloat16)
    ks = np.array([0, 5, 23, 11])
    h = torch.zeros(len(ks), D, dtype=torch.bfloat16)
    h[np.arange(len(ks)), ks] = 1.0
    ids = np.array([3, 0, 49, 17])
    st = lambda t: t.view(torch.int16).numpy().view(np.uint16)
    lse, logp, H = oracle.lmhead_row_stats(st(h), st(w), ids, "bf16", threads=1)
    wf = w.double().numpy()
    for r, k in enumerate(ks):
        col = wf[:, k]
        ref_lse = logsumexp(col)
        p = np.exp(col - ref_lse)
        assert abs(lse[r] - ref_lse) < 1e-12
        assert abs(logp[r] - (col[ids[r]] - ref_lse)) < 1e-12
        assert abs(H[r] + np.sum(p * np.log(p))) < 1e-12


def test_lmhead_policy_loss_chain_rule_finite_differences():
    """The oracle's gradients with respect to the hidden states and the LM-head
    weight are the derivatives of its own loss: central differences of the
    fp64 loss of hidden @ W^T in single entries of hidden and of W, with
    clipped tokens, the KL and entropy terms and a sequence-mean aggregation.
    A transposed product, a dropped term or a wrong sign fails this."""
    rng = np.random.default_rng(93)
    R, D, V, T = 6, 5, 11, 3
    h = rng.normal(0, 1.0, (R, D))
    W = rng.normal(0, 0.8, (V, D))
    ids = rng.integers(0, V, R)
    mask = np.array([1, 1, 0, 1, 1, 1], np.uint8)
    adv = rng.normal(0, 1, R)
    _, logp, _ = oracle.row_stats(h @ W.T, "f64", V, ids, mask, threads=1)
    lo = logp + np.array([0.3, -0.25, 0.0, 0.02, -0.4, 0.1])   # some ratios beyond the clip
    rf = logp + rng.normal(0, 0.2, R)
    kw = dict(eps=0.2, beta=0.1, c_ent=0.05, agg="seq_mean_token_mean", T=T, threads=1)
    base = oracle.lmhead_policy_loss(h, W, "f64", ids, mask, adv, lo, rf, **kw)
    assert base["clipped"].any()
    r = base["r"][mask != 0]
    assert np.min(np.abs(np.concatenate([r - 0.8, r - 1.2]))) > 1e-3  # away from the kinks

    def loss(hh, WW):
        return oracle.lmhead_policy_loss(hh, WW, "f64", ids, mask, adv, lo, rf, **kw)["loss"]

    step = 1e-6
    for (i, j) in ((0, 0), (1, 3), (2, 2), (4, 4), (5, 1)):
        hp, hm = h.copy(), h.copy()
        hp[i, j] += step
        hm[i, j] -= step
        fd = (loss(hp, W) - loss(hm, W)) / (2 * step)
        assert abs(fd - base["dhidden"][i, j]) < 1e-7, ("dhidden", i, j, fd, base["dhidden"][i, j])
    for (v, j) in ((0, 0), (int(ids[0]), 2), (7, 4), (10, 1), (int(ids[4]), 3)):
        Wp, Wm = W.copy(), W.copy()
        Wp[v, j] += step
        Wm[v, j] -= step
        fd = (loss(h, Wp) - loss(h, Wm)) / (2 * step)
        assert abs(fd - base["dweight"][v, j]) < 1e-7, ("dweight", v, j, fd, base["dweight"][v, j])
    assert np.all(base["dhidden"][2] == 0)  # a masked row has no gradient
