"""Seeded synthetic inputs for the policy-loss step.

This module draws random numbers and nothing else: it holds none of the
method's arithmetic (no softmax, no advantage, no loss), so both the CUDA path
and the CPU oracle can take their inputs from it.  Compositions that need the
method (``logp_old = logp + noise``) are made by the caller from the noise
arrays drawn here.

The workloads stand in for the rollouts the RL.cu pages train on (Qwen3-0.6B
GRPO on the mlllm.io article, "Что произошло"; PPO at batch 32 x seq 1024 in
the ainews.cool benchmark table), which are not available: the shapes are
those rollouts' shapes (vocabulary 151936 is Qwen3's), the values are draws
from the stated distributions.

Layout: sequences are group-major (sequence i = prompt * group + j); row
``b * T + t`` holds position t of sequence b; ``mask[b, t] = t < lengths[b]``.
Logits are drawn in float32 as N(0, sd) from a torch generator seeded per
block of 256 rows, then rounded (round to nearest even) to the workload's
element type, so any row range can be regenerated on its own and a given
device always yields the same bytes.
"""
from __future__ import annotations

from dataclasses import dataclass, replace

import numpy as np

ROW_BLOCK = 256


@dataclass(frozen=True)
class Workload:
    name: str
    n_prompts: int
    group: int
    T: int
    V: int
    dtype: str            # "f32" | "bf16" | "f16"
    logit_sd: float
    lengths: tuple        # ("uniform", lo, hi) | ("geometric", mean, cap) | ("full",)
    rewards: tuple        # ("bernoulli", p) | ("uniform",) | ("terminal_normal", sd)
    eps: float
    beta: float
    c_ent: float
    seed: int
    advantage: str = "group"   # "group" (GRPO) | "gae" (PPO)
    gamma: float = 1.0
    lam: float = 0.95
    value_sd: float = 0.5
    old_sd: float = 0.05
    ref_sd: float = 0.1

    @property
    def B(self) -> int:
        return self.n_prompts * self.group

    @property
    def R(self) -> int:
        return self.B * self.T

    @property
    def elem_bytes(self) -> int:
        return {"f32": 4, "bf16": 2, "f16": 2}[self.dtype]

    def scaled(self, **kw) -> "Workload":
        return replace(self, **kw)


WORKLOADS = {
    "tiny_grpo": Workload("tiny_grpo", 2, 4, 16, 1024, "f32", 2.0, ("uniform", 4, 16),
                          ("bernoulli", 0.5), 0.2, 0.04, 0.01, 101),
    "qwen3_0p6b_grpo": Workload("qwen3_0p6b_grpo", 4, 8, 1024, 151936, "bf16", 3.0,
                                ("uniform", 256, 1024), ("uniform",), 0.2, 0.04, 0.0, 102),
    "long_seq_grpo": Workload("long_seq_grpo", 2, 8, 4096, 32000, "f16", 2.0,
                              ("geometric", 1500, 4096), ("bernoulli", 0.3), 0.2, 0.0, 0.01, 103),
    "ppo_gae": Workload("ppo_gae", 64, 1, 512, 151936, "bf16", 3.0, ("full",),
                        ("terminal_normal", 1.0), 0.2, 0.0, 0.01, 104, advantage="gae"),
    "large_grpo": Workload("large_grpo", 8, 8, 2048, 151936, "bf16", 3.0,
                           ("uniform", 128, 2048), ("bernoulli", 0.5), 0.2, 0.04, 0.0, 105),
}


def small_inputs(w: Workload) -> dict:
    """Per-sequence and per-token arrays (numpy, host).

    lengths int32[B], mask uint8[R], ids int64[R], rewards float32[B] (or
    [B, T] for per-token rewards), values float32[B, T] or None, and the two
    noise draws noise_old ~ N(0, old_sd), noise_ref ~ N(0, ref_sd), float64[R].
    """
    rng = np.random.Generator(np.random.PCG64(w.seed))
    B, T = w.B, w.T
    kind = w.lengths[0]
    if kind == "uniform":
        lengths = rng.integers(w.lengths[1], w.lengths[2], size=B, endpoint=True)
    elif kind == "geometric":
        lengths = np.minimum(rng.geometric(1.0 / w.lengths[1], size=B), w.lengths[2])
    elif kind == "full":
        lengths = np.full(B, T)
    else:
        raise ValueError(kind)
    lengths = np.clip(lengths, 0, T).astype(np.int32)
    mask = (np.arange(T)[None, :] < lengths[:, None]).astype(np.uint8).reshape(-1)
    ids = rng.integers(0, w.V, size=B * T, dtype=np.int64)
    values = None
    rk = w.rewards[0]
    if rk == "bernoulli":
        rewards = (rng.random(B) < w.rewards[1]).astype(np.float32)
    elif rk == "uniform":
        rewards = rng.random(B).astype(np.float32)
    elif rk == "terminal_normal":
        rewards = np.zeros((B, T), np.float32)
        term = rng.normal(0.0, w.rewards[1], size=B).astype(np.float32)
        for b in range(B):
            if lengths[b] > 0:
                rewards[b, lengths[b] - 1] = term[b]
        values = rng.normal(0.0, w.value_sd, size=(B, T)).astype(np.float32)
    else:
        raise ValueError(rk)
    noise_old = rng.normal(0.0, w.old_sd, size=B * T)
    noise_ref = rng.normal(0.0, w.ref_sd, size=B * T)
    return dict(lengths=lengths, mask=mask, ids=ids, rewards=rewards, values=values,
                noise_old=noise_old, noise_ref=noise_ref)


def _torch_dtype(name: str):
    import torch
    return {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}[name]


def logits_block(w: Workload, block: int, device="cpu"):
    """Rows [block*256, min(R, block*256+256)) as a torch tensor of w.dtype."""
    import torch
    r0 = block * ROW_BLOCK
    n = min(w.R, r0 + ROW_BLOCK) - r0
    gen = torch.Generator(device=device)
    gen.manual_seed(w.seed * 1_000_003 + block)
    x = torch.randn((n, w.V), generator=gen, device=device, dtype=torch.float32)
    x.mul_(w.logit_sd)
    return x.to(_torch_dtype(w.dtype))


def fill_logits(w: Workload, out, row0: int = 0, row1: int | None = None, device=None):
    """Write rows [row0, row1) of the workload's logits into ``out[:, :V]``.

    ``out`` is a 2-D torch tensor [row1 - row0, ld >= V] of the workload's
    type (its padding columns are left as they are).
    """
    row1 = w.R if row1 is None else row1
    device = out.device if device is None else device
    b0, b1 = row0 // ROW_BLOCK, (row1 - 1) // ROW_BLOCK
    for b in range(b0, b1 + 1):
        blk = logits_block(w, b, device)
        lo = max(row0, b * ROW_BLOCK)
        hi = min(row1, b * ROW_BLOCK + blk.shape[0])
        out[lo - row0:hi - row0, :w.V].copy_(blk[lo - b * ROW_BLOCK:hi - b * ROW_BLOCK])
    return out


def logits(w: Workload, device="cpu", ld: int | None = None):
    """The whole logits tensor [R, ld] (padding columns zero)."""
    import torch
    ld = w.V if ld is None else ld
    out = (torch.zeros if ld != w.V else torch.empty)((w.R, ld), dtype=_torch_dtype(w.dtype),
                                                     device=device)
    if w.R:
        fill_logits(w, out)
    return out


def lmhead_inputs(R: int, D: int, V: int, seed: int, logit_sd: float = 2.0, ld_h: int | None = None,
                  ld_w: int | None = None):
    """Host torch bf16 tensors for the LM-head path: hidden [R, ld_h] with
    entries N(0, 1), weight [V, ld_w] with entries N(0, logit_sd^2 / D), both
    drawn in float32 and rounded to bf16 (padding columns past D are zero),
    and ids int64 [R] uniform on [0, V).  hidden @ weight^T then has entries
    of standard deviation about logit_sd, the spread of the logits above."""
    import torch
    ld_h = D if ld_h is None else ld_h
    ld_w = D if ld_w is None else ld_w
    gen = torch.Generator().manual_seed(seed)
    hidden = torch.zeros((R, ld_h), dtype=torch.bfloat16)
    hidden[:, :D] = torch.randn((R, D), generator=gen).to(torch.bfloat16)
    weight = torch.zeros((V, ld_w), dtype=torch.bfloat16)
    weight[:, :D] = (torch.randn((V, D), generator=gen) * (logit_sd / D ** 0.5)).to(torch.bfloat16)
    ids = torch.randint(0, V, (R,), generator=gen, dtype=torch.int64)
    return hidden, weight, ids
