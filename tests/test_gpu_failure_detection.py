"""Failure detection on the GPU without a fault: a bounded on-chip wait that
runs out reports RL_DEVERR_TIMEOUT and returns, and the CUDA context stays
usable for the next call (the same wait every kernel of the library uses)."""
import numpy as np
import pytest
import torch

import ppo_policy_loss_gb300 as rl
from ppo_policy_loss_gb300 import synth, torch_api

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    rl.build()
    rl.load()


def test_bounded_wait_times_out_and_the_context_stays_usable():
    dev = torch.device("cuda:0")
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    waited = torch.zeros(1, dtype=torch.int64, device=dev)
    limit = 50_000_000  # 50 ms
    rl.rl_selftest_wait_timeout(limit, status, waited)
    torch.cuda.synchronize()
    assert int(status.item()) & rl.RL_DEVERR_TIMEOUT
    w = int(waited.item())
    assert limit <= w < 20 * limit, w
    # the context still runs work: a small loss call succeeds and reports no error
    w_ = synth.WORKLOADS["tiny_grpo"]
    small = synth.small_inputs(w_)
    logits = synth.logits(w_, device=dev)
    t = lambda x: torch.from_numpy(np.ascontiguousarray(x)).to(dev)
    out = torch_api.policy_loss(logits, t(small["ids"]), t(small["mask"]),
                                t(np.ones(w_.B, np.float32)), w_.B, w_.T)
    st = torch_api.read_stats(out["stats"])
    assert st["device_error"] == 0 and st["n_tokens"] == int(small["mask"].sum())
