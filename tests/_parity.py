"""Shared helpers for the GPU parity tests: build inputs, run both sides, compare.

Inputs come from ppo_policy_loss_gb300.synth; the oracle's inputs are host
copies of the same bytes.  The behaviour-policy and reference log-probs are
the ORACLE's logp plus the drawn noise (never the GPU's).
"""
from __future__ import annotations

import math

import numpy as np
import torch

import oracle
from ppo_policy_loss_gb300 import synth

# ---------------------------------------------------------------- tolerances
LOGP_ATOL = 2e-3          # per-token logp and entropy, absolute
LOSS_RTOL = 1e-4          # scalar loss and the masked means, relative
LOSS_ATOL_FLOOR = 1e-7    # absolute floor when |value| < 1e-3
ADV_TOL = 1e-5            # advantages / GAE: |d| <= 1e-5 * max(|ref|, 1)
DLOGIT_ATOL = 1e-6
# fp32 dlogits (the statement fixes no fp32 tolerance): 4 fp32 ulps + 1e-6.
# The kernel keeps each row's lse, logp and exponent offset in two fp32 words
# and takes exp2f, so an element carries exp2f's error plus the rounding of
# its own exponent x (ln 2 ulp(x) relative, |x| = |log2 p|) and the sampled
# id's element r's error (expf of a two-word difference): a few ulps where
# the ulp term is the larger one; measured at most 5.6 ulps there and 6.7e-7
# absolute overall.  bf16 and fp16 outputs take 1 ulp of theirs.
DLOGIT_F32_ULPS = 4.0
CLIP_BAND = 1e-4          # |r - (1 +/- eps)| below this: clip decision may flip


def storage_np(t: torch.Tensor) -> np.ndarray:
    """Host numpy view of a tensor's element storage (uint16 for bf16/f16)."""
    t = t.detach().contiguous().cpu()
    if t.dtype in (torch.bfloat16, torch.float16):
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def adv_rows(w, small, T=None):
    """Per-row advantage from the oracle (group advantages or GAE)."""
    T = w.T if T is None else T
    if w.advantage == "gae":
        A, _ = oracle.gae(small["rewards"], small["values"], small["lengths"], w.gamma, w.lam)
        return A.reshape(-1), A
    A = oracle.group_advantages(small["rewards"], w.group)
    return np.repeat(A, T), A


def oracle_stats_chunked(logits_t, dtype, V, ids, mask, chunk=2048):
    """Oracle (lse, logp, H) for every row, copying only valid rows to the host."""
    R = mask.size
    lse, logp, ent = np.zeros(R), np.zeros(R), np.zeros(R)
    idx = np.nonzero(mask)[0]
    for i0 in range(0, idx.size, chunk):
        sel = idx[i0:i0 + chunk]
        host = storage_np(logits_t.index_select(0, torch.from_numpy(sel).to(logits_t.device))[:, :V])
        l, p, h = oracle.row_stats(host, dtype, V, ids[sel], np.ones(sel.size, np.uint8))
        lse[sel], logp[sel], ent[sel] = l, p, h
    return lse, logp, ent


def ref_rows(ref, rows):
    """The oracle's per-token gradient coefficients of the listed rows."""
    return {k: ref[k][rows] for k in ("g", "g_unclipped", "g_clipped")}


def band_mask(o, eps):
    r = o["r"]
    return (np.abs(r - (1 + eps)) < CLIP_BAND) | (np.abs(r - (1 - eps)) < CLIP_BAND)


def assert_scalar_close(name, got, ref):
    tol = LOSS_RTOL * abs(ref)
    if abs(ref) < 1e-3:
        tol = max(tol, LOSS_ATOL_FLOOR)
    assert abs(got - ref) <= tol, f"{name}: gpu {got!r} oracle {ref!r} (|d| {abs(got - ref):.3g} > {tol:.3g})"


def assert_stats_match(st, ref, n_band=0):
    """Scalars within LOSS_RTOL; counts bit-exact (n_clipped up to the n_band
    valid tokens whose ratio lies within CLIP_BAND of a clip boundary)."""
    assert st["device_error"] == 0, st
    assert st["n_tokens"] == ref["n_tokens"]
    assert abs(st["n_clipped"] - ref["n_clipped"]) <= n_band, (st["n_clipped"], ref["n_clipped"], n_band)
    for k in ("loss", "pg_term", "kl_term", "ent_term"):
        assert_scalar_close(k, st[k], ref[k])


def assert_rows_close(logp_gpu, H_gpu, ref, mask):
    mb = mask.astype(bool)
    assert np.all(logp_gpu[~mb] == 0) and np.all(H_gpu[~mb] == 0)
    dl = np.abs(logp_gpu[mb] - ref["logp"][mb])
    dh = np.abs(H_gpu[mb] - ref["entropy"][mb])
    assert dl.size == 0 or dl.max() <= LOGP_ATOL, f"logp max err {dl.max():.3g}"
    assert dh.size == 0 or dh.max() <= LOGP_ATOL, f"entropy max err {dh.max():.3g}"
    return (dl.max() if dl.size else 0.0), (dh.max() if dh.size else 0.0)


def assert_dlogits_close(gpu_store, ref_store, dtype, where=""):
    g = oracle.decode(gpu_store, dtype)
    r = oracle.decode(ref_store, dtype)
    tol = (DLOGIT_F32_ULPS if dtype == "f32" else 1.0) * oracle.ulp(r, dtype) + DLOGIT_ATOL
    err = np.abs(g - r)
    bad = ~(err <= tol)
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(f"{where} dlogits: {int(bad.sum())} elements out of tolerance; first at "
                             f"{tuple(i)}: gpu {g[tuple(i)]!r} oracle {r[tuple(i)]!r} tol {tol[tuple(i)]!r}")
    return float((err / np.maximum(oracle.ulp(r, dtype), 1e-300)).max()) if err.size else 0.0


_FMT = {"f32": (24, -126), "bf16": (8, -126), "f16": (11, -14)}


def _widen(t: torch.Tensor, dtype) -> torch.Tensor:
    """Elements of a bf16/f16/f32 tensor (or of its uint16/int16 storage) as fp64."""
    if dtype in ("bf16", "f16") and t.dtype in (torch.int16, torch.uint16):
        t = t.view(torch.int16).view(torch.bfloat16 if dtype == "bf16" else torch.float16)
    return t.float().double()


def _ulp_dev(r: torch.Tensor, dtype) -> torch.Tensor:
    """oracle.ulp on the device: the spacing of ``dtype`` at |r| (r holds values
    of that format), built from the fp32 exponent field so that it is exact."""
    p, emin = _FMT[dtype]
    bits = r.abs().float().view(torch.int32)
    e = ((bits >> 23) & 0xFF).to(torch.int64) - 127      # -127 for 0 and fp32 subnormals
    u = torch.clamp(e, min=emin) - (p - 1)
    return ((u + 1023) << 52).view(torch.float64)


def rows_within(gpu_rows: torch.Tensor, ref_store: np.ndarray, dtype):
    """Per row: True when every element of the GPU's gradient row lies within
    the dlogits tolerance of the oracle's rounded value.  Compared on the
    device (the full-size workloads hold tens of GB of gradient).  Returns
    (per-row bool array, max error in units of the oracle value's ulp)."""
    dev = gpu_rows.device
    ref = torch.from_numpy(np.ascontiguousarray(ref_store))
    if dtype in ("bf16", "f16"):
        ref = ref.view(torch.int16)
    r = _widen(ref.to(dev), dtype)
    g = _widen(gpu_rows, dtype)
    u = _ulp_dev(r, dtype)
    tol = (DLOGIT_F32_ULPS if dtype == "f32" else 1.0) * u + DLOGIT_ATOL
    err = (g - r).abs()
    ok = (err <= tol).all(dim=1)          # NaN compares false
    worst = float((err / u).max()) if err.numel() else 0.0
    return ok.cpu().numpy(), worst


def check_dlogits_rows(gpu_rows, host, dtype, V, ids, rows, lse, ent, ref, band, scale, c_ent,
                       where=""):
    """Every listed row of the GPU's gradient against the oracle.

    ``host`` holds the logits storage that ``rows`` index (with ``ids``);
    ``lse``, ``ent``, ``scale`` and ``band`` are per listed row, ``ref`` is the
    oracle's loss_from_stats output indexed by the same listed rows.  A row
    in the clip band (its ratio within CLIP_BAND of a clip boundary, where
    the kernel's fp32 ratio may fall on the other side) must match the
    gradient of one of the surrogate's two branches; every other row must
    match the oracle's own gradient.  Returns the max error in ulps."""
    main = oracle.dlogits_rows(host, dtype, V, ids, rows, lse, ent, ref["g"], scale, c_ent, dtype)
    ok, worst = rows_within(gpu_rows, main, dtype)
    for i in np.nonzero(~ok & band)[0]:  # a band row may take the other branch
        for key in ("g_unclipped", "g_clipped"):
            alt = oracle.dlogits_rows(host, dtype, V, ids, rows[i:i + 1], lse[i:i + 1],
                                      ent[i:i + 1], ref[key][i:i + 1], scale[i:i + 1], c_ent, dtype)
            if rows_within(gpu_rows[i:i + 1], alt, dtype)[0][0]:
                ok[i] = True
                break
    if not ok.all():
        i = int(np.nonzero(~ok)[0][0])
        g = _widen(gpu_rows[i:i + 1], dtype).cpu().numpy()[0]
        r = oracle.decode(main[i], dtype)
        j = int(np.argmax(np.abs(g - r)))
        raise AssertionError(f"{where} dlogits: {int((~ok).sum())} of {ok.size} rows out of "
                             f"tolerance; first: listed row {i} (band {bool(band[i])}), element "
                             f"{j}: gpu {g[j]!r} oracle {r[j]!r}")
    return worst


def build_case(w, device="cuda", ld=None, n_rows=None):
    """Inputs for workload w (optionally only its first n_rows rows, T kept)."""
    small = synth.small_inputs(w)
    V = w.V
    ld = V if ld is None else ld
    logits = synth.logits(w, device=device, ld=ld)
    if n_rows is not None:
        logits = logits[:n_rows].contiguous() if ld == V else logits[:n_rows]
    return small, logits


def composed_old_ref(logp_oracle, small, mask, R):
    """logp_old = oracle logp + N(0, old_sd); ref = oracle logp + N(0, ref_sd); stored fp32."""
    lo = (logp_oracle + small["noise_old"][:R]).astype(np.float32)
    rf = (logp_oracle + small["noise_ref"][:R]).astype(np.float32)
    lo[mask == 0] = 0.0
    rf[mask == 0] = 0.0
    return lo, rf


def to_dev(x, device="cuda"):
    return torch.from_numpy(np.ascontiguousarray(x)).to(device)


def valid_and_masked_sample(mask, k, seed=0):
    rng = np.random.default_rng(seed)
    v = np.nonzero(mask)[0]
    m = np.nonzero(mask == 0)[0]
    pick = list(rng.choice(v, size=min(k, v.size), replace=False)) if v.size else []
    pick += list(rng.choice(m, size=min(max(1, k // 4), m.size), replace=False)) if m.size else []
    if v.size:
        pick += [int(v[0]), int(v[-1])]
    return np.unique(np.array(pick, np.int64))


def rel(a, b):
    return abs(a - b) / max(abs(b), 1e-30)


def ceil_div(a, b):
    return -(-a // b)


__all__ = [n for n in dir() if not n.startswith("_")] + ["math"]


def accumulation_bound(A: np.ndarray, B: np.ndarray, block: int = 16, u: float = 2.0 ** -24):
    """Element-wise bound on |C - A @ B| for C an fp32 accumulation of the exact
    products of A [M, K] and B [K, N] (fp64 arrays of 16-bit values, whose
    products are exact in fp32), in K order, one block of `block` products
    per step.  Each step rounds the running sum once: the error is at most u
    times the sum of the magnitudes of the running sums after each step
    (recursive summation), plus u times the sum of the products' magnitudes
    for the rounding inside a step; both are doubled, allowing a unit that
    truncates instead of rounding to nearest."""
    K = A.shape[1]
    S = np.zeros((A.shape[0], B.shape[1]))
    run = np.zeros_like(S)
    for k0 in range(0, K, block):
        S += A[:, k0:k0 + block] @ B[k0:k0 + block]
        run += np.abs(S)
    return 2.0 * u * (run + np.abs(A) @ np.abs(B))
