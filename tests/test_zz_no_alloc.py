"""rl_policy_loss_fwd_bwd_noalloc: the loss entry point for callers that cannot
allocate device memory (a plug-in whose host framework owns the GPU allocator,
or a program that hands all device memory to its own pool up front).  It uses
the library's static scratch array instead of a caller workspace.

Checked through the C ABI: calls in a row, alternating between a shape of
each build of the loss kernel (so consecutive calls use grids of different
sizes), must each agree with the allocating entry point, within the
tolerances of the parity tests.  This file is
collected last so that a run stopping at the first failure has already run
every other test; it also passes on its own in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

import ppo_policy_loss_gb300 as rl
from ppo_policy_loss_gb300 import STATS_BYTES, synth, torch_api
from _parity import (LOGP_ATOL, assert_dlogits_close, assert_scalar_close, storage_np, to_dev)

pytestmark = pytest.mark.gpu


# Two shapes that take the two builds of the loss kernel with different grid
# sizes: V = 151936 bf16 rows (long-row build, one CTA per row here: 128
# CTAs) and V = 32000 fp16 rows (short-row build, two CTAs per SM: a grid of
# twice the SM count over 512 rows).
CASES = {
    "bf16": (synth.WORKLOADS["qwen3_0p6b_grpo"].scaled(n_prompts=2, group=4, T=16,
                                                       lengths=("uniform", 4, 16), c_ent=0.01),
             rl.RL_BF16),
    "f16": (synth.WORKLOADS["long_seq_grpo"].scaled(n_prompts=1, group=8, T=64,
                                                    lengths=("uniform", 8, 64), beta=0.04),
            rl.RL_F16),
}


def _inputs(w):
    small = synth.small_inputs(w)
    logits = synth.logits(w, device="cuda")
    lo = to_dev((small["noise_old"] - 12.0).astype(np.float32))
    rf = to_dev((small["noise_ref"] - 12.0).astype(np.float32))
    adv = torch_api.group_advantages(to_dev(small["rewards"]), w.group)
    return logits, to_dev(small["ids"]), to_dev(small["mask"]), adv, lo, rf


def _outputs(w, logits):
    return (torch.empty_like(logits), torch.empty(w.R, device="cuda"),
            torch.empty(w.R, device="cuda"), torch.zeros(STATS_BYTES, dtype=torch.uint8,
                                                         device="cuda"))


def test_noalloc_matches_allocating_entry_point_twice():
    rl.build()
    lib = rl.load()
    stream = torch.cuda.current_stream().cuda_stream
    runs = {}
    keep = []  # the calls below take raw device pointers: keep every input tensor alive
    for name, (w, code) in CASES.items():
        logits, ids, mask, adv, lo, rf = _inputs(w)
        keep.append((ids, mask, adv, lo, rf))
        common = (logits.data_ptr(), code, w.B, w.T, w.V, w.V, ids.data_ptr(), lo.data_ptr(),
                  rf.data_ptr(), mask.data_ptr(), adv.data_ptr(), rl.RL_ADV_PER_SEQ,
                  ctypes.c_float(w.eps), ctypes.c_float(w.beta), ctypes.c_float(w.c_ent),
                  ctypes.c_float(float(int(mask.sum()))))
        # the allocating entry point, with a caller workspace
        d_ref, lp_ref, h_ref, st_ref = _outputs(w, logits)
        ws = torch.zeros(rl.rl_policy_loss_workspace_size(w.R), dtype=torch.uint8, device="cuda")
        assert lib.rl_policy_loss_fwd_bwd(*common, d_ref.data_ptr(), lp_ref.data_ptr(),
                                          h_ref.data_ptr(), st_ref.data_ptr(), ws.data_ptr(),
                                          ws.numel(), stream) == rl.RL_OK
        torch.cuda.synchronize()
        ref = torch_api.read_stats(st_ref)
        assert ref["device_error"] == 0 and ref["n_tokens"] > 0
        runs[name] = (w, logits, common, d_ref, lp_ref, h_ref, ref)

    # Alternate the two shapes: each call finds the previous call's contents,
    # left by a grid of another size, in the scratch.
    for call, name in enumerate(["bf16", "f16", "bf16", "f16"]):
        w, logits, common, d_ref, lp_ref, h_ref, ref = runs[name]
        d, lp, h, st = _outputs(w, logits)
        assert lib.rl_policy_loss_fwd_bwd_noalloc(*common, d.data_ptr(), lp.data_ptr(),
                                                  h.data_ptr(), st.data_ptr(), stream) == rl.RL_OK
        torch.cuda.synchronize()
        got = torch_api.read_stats(st)
        assert got["device_error"] == 0, (call, name, got)
        assert got["n_tokens"] == ref["n_tokens"] and got["n_clipped"] == ref["n_clipped"]
        for k in ("loss", "pg_term", "kl_term", "ent_term"):
            assert_scalar_close(k, got[k], ref[k])
        assert float((lp - lp_ref).abs().max()) <= LOGP_ATOL
        assert float((h - h_ref).abs().max()) <= LOGP_ATOL
        assert_dlogits_close(storage_np(d), storage_np(d_ref), w.dtype,
                             where=f"noalloc call {call} ({name})")
