"""Benchmark of the fused RL policy-loss step on GB300.

One step = the whole hot path over one batch: the advantages (GRPO reward
normalisation with rl_group_advantages, or PPO-GAE with rl_gae_reverse_scan)
then rl_policy_loss_fwd_bwd (log-softmax, clipped surrogate, k3 KL, entropy
bonus, masked-mean loss and the logits gradient in one launch).

Default workload (the headline): Qwen3-0.6B-shaped GRPO, 4 prompts x group 8
= 32 sequences x T=1024 positions x V=151936 bf16 logits ~N(0, 3), ragged
lengths U{256..1024}; synthetic seeded inputs; 10 GB of logits, far larger
than L2, so no flush is needed between steps.  ``--workload`` selects one of
the other configurations (see ppo_policy_loss_gb300/synth.py).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
                    [--workload NAME] [--lmhead]

Prints one JSON line (rank 0).  With N > 1 (torchrun) every rank runs its own
batch of the workload on its GPU (weak scaling); by default each rank's loss
is normalised by its own tokens (independent replicas, no collective on the
data path), and with ``--global-token-mean`` by the tokens of all ranks (the
path's one exchange: an all-reduce of the token counts before the loss and
of the loss shares after).  value = all ranks' tokens / max-over-ranks time.
``--impl reference`` times the fp64 CPU oracle instead, on a bounded sample
of the same workload.

``--lmhead`` times the other tensor-core path instead: rl_lmhead_logprobs on
the Qwen3-0.6B LM head (D=1024, V=151936 bf16) over the same 32 x 1024 rows,
i.e. the policy's log-probs of the sampled tokens straight from the hidden
states, with a tensor-core roofline (2 R D V flops per launch).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "fused GRPO loss+dlogits tokens/s at V=151936 bf16; % of HBM roofline"
WORKLOAD = "qwen3_0p6b_grpo"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
LMHEAD_METRIC = "fused LM-head + log-softmax rows/s (Qwen3 head, V=151936 bf16); % of tensor roofline"
LMHEAD_SHAPE = dict(R=32 * 1024, D=1024, V=151936, logit_sd=3.0, seed=202)
KERNEL_SRC = os.path.join(ROOT, "ppo_policy_loss_gb300", "csrc", "policy_loss.cu")
# the loss kernel's translation unit: its source and the headers of this
# project that it includes
KERNEL_SRCS = (KERNEL_SRC, os.path.join(ROOT, "ppo_policy_loss_gb300", "csrc", "rl_device.cuh"),
               os.path.join(ROOT, "include", "rlloss.h"))
LMHEAD_SRC = os.path.join(ROOT, "ppo_policy_loss_gb300", "csrc", "lmhead.cu")
# the workloads timed after the headline (their kernel times and roofline
# fractions go into the line's "workloads" object)
OTHER_WORKLOADS = ("ppo_gae", "large_grpo", "long_seq_grpo", "tiny_grpo")
DESCRIBE = {
    "tiny_grpo": "tiny GRPO: 2 prompts x group 4 = 8 seqs, T=16, V=1024 fp32",
    "qwen3_0p6b_grpo": "Qwen3-0.6B GRPO: 4 prompts x group 8 = 32 seqs, T=1024, V=151936 bf16, "
                       "lengths U{256..1024}, eps=0.2 beta=0.04 c_ent=0",
    "long_seq_grpo": "long-sequence GRPO: 2 prompts x group 8 = 16 seqs, T=4096, V=32000 fp16, "
                     "geometric lengths (mean 1500, cap 4096), beta=0 c_ent=0.01",
    "ppo_gae": "PPO-GAE: 64 seqs, T=512, V=151936 bf16, gamma=1 lambda=0.95, c_ent=0.01",
    "large_grpo": "large GRPO: 8 prompts x group 8 = 64 seqs, T=2048, V=151936 bf16, "
                  "lengths U{128..2048}, eps=0.2 beta=0.04",
}


def traffic_file(workload):
    return os.path.join(ROOT, "profiles", f"policy_loss_{workload}_traffic.txt")


# ----------------------------------------------------------------------------- helpers
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def bf16_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return float(json.load(f)["bf16_tflops"]), "measured (burst)"
    except Exception:
        return FALLBACK_BF16_TFLOPS, "fallback"


def bf16_sustained_peak():
    """The bf16 GEMM rate held for seconds under the power cap, or None."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return float(json.load(f)["bf16_tflops_sustained"])
    except Exception:
        return None


def hbm_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def code_only(text: str) -> str:
    """C/C++/CUDA source without its comments, trailing blanks and blank
    lines (the kernel's files hold no comment markers inside string
    literals)."""
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    lines = (re.sub(r"//.*", "", line).rstrip() for line in text.splitlines())
    return "\n".join(line for line in lines if line)


def kernel_sha(src=None) -> str:
    """First 16 hex digits of the sha256 of the loss kernel's code (`src`: a
    path or a sequence of paths, by default its translation unit), comments
    and blank lines left out: a change to the code gives a new value, an edit
    to comments alone keeps the records taken on the kernel valid."""
    paths = KERNEL_SRCS if src is None else ((src,) if isinstance(src, str) else tuple(src))
    h = hashlib.sha256()
    for path in paths:
        with open(path, encoding="utf-8") as f:
            h.update(code_only(f.read()).encode())
        h.update(b"\0")
    return h.hexdigest()[:16]


def recorded_traffic(workload=WORKLOAD, path=None, src=None):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the current kernel source; else None."""
    try:
        kv = {}
        with open(path or traffic_file(workload)) as f:
            for line in f:
                if ":" in line and not line.startswith("#"):
                    k, v = line.split(":", 1)
                    kv[k.strip()] = v.strip()
        if kv.get("kernel_sha") != kernel_sha(src):
            return None
        return float(kv["dram_bytes_per_launch"])
    except Exception:
        return None


def max_over_ranks(x: float, device) -> float:
    """Max of a per-rank scalar over all ranks (identity when not distributed)."""
    import torch
    import torch.distributed as dist
    if not dist.is_available() or not dist.is_initialized() or dist.get_world_size() == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(rows_per_rank: int, world: int, ms_per_step: float) -> float:
    """Positions per second over all ranks: every rank runs its own replica."""
    return world * rows_per_rank / (ms_per_step / 1e3)


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 200 ms."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.file = None

    def start(self):
        self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.file, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        self.proc.wait()
        self.file.flush()
        self.file.seek(0)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.file:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        os.unlink(self.file.name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "samples": len(sm), "reasons": sorted(reasons)}


# ----------------------------------------------------------------------------- inputs
def make_inputs(w, dev):
    """Device inputs of the workload.  logp_old / ref_logp are composed from the
    current policy's own log-probs (computed once here with torch, untimed) plus
    the workload's noise draws."""
    import torch
    from ppo_policy_loss_gb300 import synth

    small = synth.small_inputs(w)
    logits = synth.logits(w, device=dev)

    def t(x, dt=None):
        a = torch.from_numpy(np.ascontiguousarray(x)).to(dev)
        return a if dt is None else a.to(dt)

    inp = dict(small=small, logits=logits, ids=t(small["ids"]), mask=t(small["mask"]),
               rewards=t(small["rewards"]))
    if w.advantage == "gae":
        inp["values"] = t(small["values"])
        inp["lengths"] = t(small["lengths"])
    logp = torch.empty(w.R, dtype=torch.float32, device=dev)
    for r0 in range(0, w.R, 1024):  # torch log_softmax, chunked (input preparation only)
        blk = logits[r0:r0 + 1024].float()
        lse = torch.logsumexp(blk, dim=1)
        logp[r0:r0 + 1024] = blk.gather(1, inp["ids"][r0:r0 + 1024, None])[:, 0] - lse
        del blk
    m = inp["mask"].bool()
    inp["logp_old"] = torch.where(m, logp + t(small["noise_old"], torch.float32), 0.0).contiguous()
    inp["ref"] = torch.where(m, logp + t(small["noise_ref"], torch.float32), 0.0).contiguous()
    return inp


def alg_bytes(w, n_valid):
    """Algorithmic bytes of one rl_policy_loss_fwd_bwd launch: one read of each
    valid logits row, one write of every dlogits row, plus the per-row arrays
    (ids 8, logp_old 4, ref 4 when the KL term is on, mask 1, logp_out 4,
    entropy_out 4) and the advantages (per sequence, or per token for PPO-GAE)."""
    es = w.elem_bytes
    adv = w.R * 4 if w.advantage == "gae" else w.B * 4
    ref = 4 if w.beta != 0 else 0
    return n_valid * w.V * es + w.R * w.V * es + w.R * (8 + 4 + ref + 1 + 4 + 4) + adv


class Step:
    """Device buffers of one step and the launches of the whole path on them."""

    KEYS = ("logits", "ids", "mask", "rewards", "logp_old", "ref", "values", "lengths")

    def __init__(self, w, inp, dev, own_inputs=False):
        import torch
        from ppo_policy_loss_gb300 import torch_api

        self.w = w
        self.keys = [k for k in self.KEYS if k in inp]
        self.d = {k: (torch.empty_like(inp[k]) if own_inputs else inp[k]) for k in self.keys}
        self.adv = torch.empty(w.R if w.advantage == "gae" else w.B, dtype=torch.float32,
                               device=dev)
        self.dlogits = torch.empty_like(inp["logits"])
        self.logp = torch.empty(w.R, dtype=torch.float32, device=dev)
        self.ent = torch.empty(w.R, dtype=torch.float32, device=dev)
        self.ws = torch_api.new_workspace(w.R, dev)
        self.stats = torch_api.new_stats(dev)
        self.ld = inp["logits"].stride(0)

    def launch(self, stream, ev=None, global_mean=False):
        """2 launches: the advantages, then the fused loss (bracketed by ev).
        With global_mean (data parallel over ranks): 3 launches and two small
        all-reduces, the token counts before the loss and its shares after."""
        import ppo_policy_loss_gb300 as rl
        w, d = self.w, self.d
        if global_mean:
            import torch.distributed as dist
            from ppo_policy_loss_gb300 import torch_api
            self.counts = torch_api.count_tokens(d["mask"], w.B, w.T, stream=stream)
            dist.all_reduce(self.counts)
        if w.advantage == "gae":
            rl.rl_gae_reverse_scan(d["rewards"], d["values"], d["lengths"], w.B, w.T, w.gamma,
                                   w.lam, self.adv, None, stream)
            layout = rl.RL_ADV_PER_TOKEN
        else:
            rl.rl_group_advantages(d["rewards"], w.B // w.group, w.group, 1e-4, 1, self.adv,
                                   stream)
            layout = rl.RL_ADV_PER_SEQ
        if ev is not None:
            ev[0].record(stream)
        if global_mean:
            desc = rl.rl_policy_loss_desc_init()
            p = lambda t: t.data_ptr() if t is not None else None
            desc.logits, desc.dtype, desc.B, desc.T, desc.V, desc.ld = (
                p(d["logits"]), rl.DTYPES[w.dtype], w.B, w.T, w.V, self.ld)
            desc.ids, desc.logp_old, desc.mask, desc.adv = (p(d["ids"]), p(d["logp_old"]),
                                                            p(d["mask"]), p(self.adv))
            desc.ref_logp = p(d["ref"]) if w.beta != 0 else None
            desc.adv_layout, desc.eps, desc.eps_high = layout, w.eps, w.eps
            desc.beta, desc.c_ent, desc.grad_scale = w.beta, w.c_ent, 1.0
            desc.dlogits, desc.logp_out, desc.entropy_out = (p(self.dlogits), p(self.logp),
                                                             p(self.ent))
            desc.stats_dev, desc.workspace, desc.workspace_bytes = (p(self.stats), p(self.ws),
                                                                    self.ws.numel())
            desc.global_counts = p(self.counts)
            rl.rl_policy_loss_fwd_bwd_ex(desc, stream)
        else:
            rl.rl_policy_loss_fwd_bwd(d["logits"], w.dtype, w.B, w.T, w.V, self.ld, d["ids"],
                                      d["logp_old"], d["ref"] if w.beta != 0 else None,
                                      d["mask"], self.adv, layout, w.eps, w.beta, w.c_ent, 1.0,
                                      self.dlogits, self.logp, self.ent, self.stats, self.ws,
                                      self.ws.numel(), stream)
        if ev is not None:
            ev[1].record(stream)
        if global_mean:
            import torch.distributed as dist
            self.loss_share = self.stats[:8].view(__import__("torch").float64).clone()
            dist.all_reduce(self.loss_share)


def workload_for(args):
    from ppo_policy_loss_gb300 import synth
    w = synth.WORKLOADS[args.workload]
    if args.seqs:  # a slice of the workload (profiling captures): same T, V and distributions
        w = (w.scaled(n_prompts=max(1, args.seqs // w.group)) if args.seqs >= w.group
             else w.scaled(n_prompts=1, group=max(2, args.seqs)))
    # other shapes of the same workload (profiling captures and sweeps)
    if getattr(args, "vocab", 0):
        w = w.scaled(V=args.vocab)
    if getattr(args, "dtype", None):
        w = w.scaled(dtype=args.dtype)
    if getattr(args, "seq_len", 0):
        w = w.scaled(T=args.seq_len)
    if getattr(args, "all_valid", False):
        w = w.scaled(lengths=("full",))
    if getattr(args, "c_ent", None) is not None:
        w = w.scaled(c_ent=args.c_ent)
    return w


def reshaped(args) -> bool:
    return bool(args.seqs or getattr(args, "vocab", 0) or getattr(args, "dtype", None)
                or getattr(args, "seq_len", 0) or getattr(args, "all_valid", False)
                or getattr(args, "c_ent", None) is not None)


# ----------------------------------------------------------------------------- GPU arm
def run_gpu(args):
    import torch

    import ppo_policy_loss_gb300 as rl
    from ppo_policy_loss_gb300 import torch_api

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    rl.build()
    rl.load()
    w = workload_for(args)
    inp = make_inputs(w, dev)
    n_valid = int(inp["small"]["mask"].sum())
    stream = torch.cuda.current_stream(dev)
    step = Step(w, inp, dev)

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize(dev)

    gm = bool(args.global_token_mean and world > 1)
    for _ in range(args.warmup):
        step.launch(stream, global_mean=gm)
    barrier()
    st = torch_api.read_stats(step.stats)
    assert st["device_error"] == 0 and st["n_tokens"] == n_valid, st

    # ---- timed region: K steps, inputs resident in HBM
    kev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    sampler = ClockSampler(int(vis.split(",")[local]) if vis else local)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    sampler.start()
    time.sleep(0.3)
    t0.record(stream)
    for i in range(args.steps):
        step.launch(stream, kev[i], global_mean=gm)
    t1.record(stream)
    barrier()
    clocks = sampler.stop()
    ms_total = max_over_ranks(t0.elapsed_time(t1), dev)
    k_ms = [a.elapsed_time(b) for a, b in kev]
    ms_step = ms_total / args.steps
    value = whole_job_rate(w.R, world, ms_step)

    # ---- roofline of the dominant kernel (rl_policy_loss_fwd_bwd)
    kern_ms = statistics.mean(k_ms)
    bytes_launch = alg_bytes(w, n_valid)
    peak, peak_kind = hbm_peak()
    achieved = bytes_launch / (kern_ms / 1e3) / 1e9
    traffic = recorded_traffic(args.workload) if not reshaped(args) else None

    # ---- end to end through the C ABI with pinned host buffers
    e2e = run_e2e(args, w, inp, dev, stream, step) if args.e2e_steps > 0 else None
    shape = rl.rl_policy_loss_launch_shape(w.dtype, w.V, w.R)
    out = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": w.dtype,
        "data": "synthetic (seeded; shapes and distributions of the workload)",
        "config": {"workload": f"{args.workload}: {DESCRIBE.get(args.workload, '')}",
                   "B": w.B, "T": w.T, "V": w.V, "rows": w.R, "valid_tokens": n_valid,
                   "slice": (f"profiling shape: {w.B} sequences x T={w.T}, V={w.V} {w.dtype}, "
                             f"lengths {w.lengths[0]}, c_ent={w.c_ent}" if reshaped(args) else None),
                   "valid_tokens_per_s": world * n_valid / (ms_step / 1e3),
                   "l2": (f"inputs ({w.R * w.V * w.elem_bytes / 1e9:.1f} GB logits) vs 129 MB "
                          "L2; no flush"),
                   "parallelism": ("data parallel, global token mean (all-reduce of the "
                                   "token counts and of the loss shares)" if gm else
                                   "replicas" if world > 1 else "single GPU"),
                   "launch_shape": {"cluster": shape[0], "clusters": shape[1],
                                    "smem": shape[2]}},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_source": peak_kind,
                     "traffic": traffic, "alg_bytes_per_launch": bytes_launch,
                     "kernel": "rl_policy_loss_fwd_bwd", "kernel_ms": kern_ms},
        "e2e": e2e,
        "aux_kernels": (time_aux(w, inp, dev, stream) if not args.no_aux else None),
        "gpu_launches": (3 if gm else 2) * args.steps,
        "clocks": clocks,
    }
    if rank == 0 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baselines(w, args.workload, inp["logits"],
                                            budget_s=args.cpu_seconds)
    if world == 1 and not args.no_workloads and not reshaped(args):
        del step, inp
        torch.cuda.empty_cache()
        out["workloads"] = {name: time_workload(name, dev, stream, args,
                                                int(vis.split(",")[local]) if vis else local)
                            for name in OTHER_WORKLOADS if name != args.workload}
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(out), flush=True)


def time_workload(name, dev, stream, args, gpu_index, min_region_s=0.6, max_steps=3000):
    """The same step on another workload, timed after the headline's timed
    region with the headline's buffers freed: warm-up, then enough steps for
    a timed region of about ``min_region_s`` (at least --steps), the loss
    launch bracketed by CUDA events, clocks sampled over the region."""
    import torch

    from ppo_policy_loss_gb300 import synth, torch_api

    w = synth.WORKLOADS[name]
    inp = make_inputs(w, dev)
    n_valid = int(inp["small"]["mask"].sum())
    step = Step(w, inp, dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for i in range(args.warmup):
        if i == args.warmup - 1:
            e0.record(stream)
        step.launch(stream)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    st = torch_api.read_stats(step.stats)
    assert st["device_error"] == 0 and st["n_tokens"] == n_valid, (name, st)
    est_ms = max(e0.elapsed_time(e1), 1e-3)
    steps = int(min(max_steps, max(args.steps, min_region_s * 1e3 / est_ms)))
    kev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    sampler = ClockSampler(gpu_index)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    sampler.start()
    time.sleep(0.3)
    t0.record(stream)
    for i in range(steps):
        step.launch(stream, kev[i])
    t1.record(stream)
    torch.cuda.synchronize(dev)
    clocks = sampler.stop()
    ms_step = t0.elapsed_time(t1) / steps
    k_ms = [a.elapsed_time(b) for a, b in kev]
    kern_ms = statistics.mean(k_ms)
    nbytes = alg_bytes(w, n_valid)
    peak, peak_kind = hbm_peak()
    achieved = nbytes / (kern_ms / 1e3) / 1e9
    in_l2 = w.R * w.V * w.elem_bytes * 2 < 64e6
    out = {"workload": f"{name}: {DESCRIBE.get(name, '')}", "B": w.B, "T": w.T, "V": w.V,
           "dtype": w.dtype, "rows": w.R, "valid_tokens": n_valid, "steps": steps,
           "ms_per_step": ms_step, "tokens_per_s": w.R / (ms_step / 1e3),
           "kernel_ms": kern_ms, "kernel_ms_min": min(k_ms), "alg_bytes_per_launch": nbytes,
           "achieved_GB_per_s": achieved, "peak": peak, "peak_source": peak_kind,
           "frac": None if in_l2 else achieved / peak,
           "bound": "latency (inputs stay in L2)" if in_l2 else "hbm",
           "traffic": recorded_traffic(name), "clocks": clocks,
           "gpu_launches": 2 * steps}
    del step, inp
    torch.cuda.empty_cache()
    return out


def time_aux(w, inp, dev, stream, reps=50):
    """Mean device time (CUDA events, `reps` back-to-back launches after a
    warm-up) of the O(B*T) kernels beside the loss, at this workload's sizes:
    group advantages, GAE, masked whitening, the critic loss and the token
    count.  GRPO workloads get seeded values and per-token rewards for the
    GAE and critic calls."""
    import torch

    import ppo_policy_loss_gb300 as rl
    from ppo_policy_loss_gb300 import VALUE_STATS_BYTES

    B, T, R = w.B, w.T, w.R
    g = torch.Generator(device=dev).manual_seed(w.seed)
    mask = inp["mask"]
    values = (inp["values"] if "values" in inp else
              0.5 * torch.randn((B, T), generator=g, device=dev)).contiguous()
    rewards_t = (inp["rewards"] if w.advantage == "gae" else
                 torch.randn((B, T), generator=g, device=dev)).contiguous()
    lengths = (inp["lengths"] if "lengths" in inp else
               mask.view(B, T).sum(1).to(torch.int32)).contiguous()
    adv_seq = torch.empty(B, device=dev)
    adv_tok, ret = torch.empty(R, device=dev), torch.empty(R, device=dev)
    white = torch.empty(R, device=dev)
    dval = torch.empty(R, device=dev)
    vst = torch.zeros(VALUE_STATS_BYTES, dtype=torch.uint8, device=dev)
    counts = torch.empty(2, dtype=torch.int64, device=dev)
    rewards_seq = (inp["rewards"] if w.advantage != "gae" else
                   torch.rand(B, generator=g, device=dev)).contiguous()
    vold = (values + 0.1 * torch.randn((B, T), generator=g, device=dev)).contiguous()
    G = w.group if w.group > 1 else (8 if B % 8 == 0 else B)  # PPO workloads: groups of 8
    calls = {
        "group_advantages": (lambda: rl.rl_group_advantages(rewards_seq, B // G, G, 1e-4, 1, adv_seq,
                                                              stream), B * 8),
        "gae_reverse_scan": (lambda: rl.rl_gae_reverse_scan(rewards_t, values, lengths, B, T, w.gamma,
                                                              w.lam, adv_tok, ret, stream),
                             R * 16 + B * 4),
        "masked_whiten": (lambda: rl.rl_masked_whiten(adv_tok, mask, R, 1e-8, 1, white, stream),
                          R * 9),
        "value_loss": (lambda: rl.rl_value_loss_fwd_bwd(values, vold, ret, mask, R, 0.2, 1.0, dval,
                                                        vst, stream), R * 17),
        "count_tokens": (lambda: rl.rl_count_tokens(mask, B, T, counts, stream), R),
    }
    out = {}
    for name, (fn, nbytes) in calls.items():
        for _ in range(3):
            fn()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(reps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        us = e0.elapsed_time(e1) * 1e3 / reps
        out[name] = {"us": round(us, 2), "bytes": nbytes, "GB_per_s": round(nbytes / us / 1e3, 1)}
    return out


def run_e2e(args, w, inp, dev, stream, step0):
    """The same step through the public C-ABI calls with HOST inputs: every
    step uploads its inputs from pinned host memory and reads its results
    (the loss statistics and the per-token log-probs and entropies) back,
    inside the timed region.  The logits gradient stays on the device, where
    the backward pass through the LM head consumes it.

    Only the logits rows the loss reads are uploaded: each sequence's valid
    prefix, one copy per sequence (masked rows are never read by the kernel;
    their device rows keep stale bytes).  The other inputs go whole.  Steps
    are double-buffered like a training loop that prefetches its next batch:
    the upload of step i+1 runs on its own stream beside the compute of step
    i, with events keeping a buffer set from being overwritten before its
    last reader is done."""
    import torch

    from ppo_policy_loss_gb300 import STATS_BYTES, stats_from_bytes

    steps = max(1, min(args.steps, args.e2e_steps))
    h = {}
    for k in step0.keys:
        h[k] = torch.empty(inp[k].shape, dtype=inp[k].dtype, pin_memory=True)
        h[k].copy_(inp[k])
    lengths = np.clip(inp["small"]["lengths"].astype(np.int64), 0, w.T)
    spans = [(b * w.T, b * w.T + int(L)) for b, L in enumerate(lengths) if L > 0]
    h_stats = torch.empty(STATS_BYTES, dtype=torch.uint8, pin_memory=True)
    h_logp = torch.empty(w.R, dtype=torch.float32, pin_memory=True)
    h_ent = torch.empty(w.R, dtype=torch.float32, pin_memory=True)
    sets = [Step(w, inp, dev, own_inputs=True), Step(w, inp, dev, own_inputs=True)]
    row_bytes = inp["logits"].stride(0) * inp["logits"].element_size()
    h2d = sum(t.numel() * t.element_size() for k, t in h.items() if k != "logits")
    h2d += sum(r1 - r0 for r0, r1 in spans) * row_bytes
    d2h = STATS_BYTES + 2 * w.R * 4
    s_in = torch.cuda.Stream(dev)
    s_cmp = stream
    comp_done = [torch.cuda.Event(), torch.cuda.Event()]  # last compute on set b finished
    for e in comp_done:
        e.record(s_cmp)

    def one(i):
        b = sets[i % 2]
        with torch.cuda.stream(s_in):
            s_in.wait_event(comp_done[i % 2])          # set b's inputs no longer read
            for k in b.keys:
                if k == "logits":
                    for r0, r1 in spans:
                        b.d[k][r0:r1].copy_(h[k][r0:r1], non_blocking=True)
                else:
                    b.d[k].copy_(h[k], non_blocking=True)
            in_done = torch.cuda.Event()
            in_done.record(s_in)
        s_cmp.wait_event(in_done)
        b.launch(s_cmp)
        h_stats.copy_(b.stats, non_blocking=True)
        h_logp.copy_(b.logp, non_blocking=True)
        h_ent.copy_(b.ent, non_blocking=True)
        comp_done[i % 2].record(s_cmp)

    one(0)
    one(1)
    torch.cuda.synchronize(dev)
    link = host_link(dev)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(s_cmp)
    s_in.wait_event(t0)
    for i in range(steps):
        one(i)
    t1.record(s_cmp)
    torch.cuda.synchronize(dev)
    ms = max_over_ranks(t0.elapsed_time(t1), dev) / steps
    world = dist_env()[0]
    st = stats_from_bytes(h_stats.numpy().tobytes())
    del sets, h
    return {"value": whole_job_rate(w.R, world, ms), "unit": "tokens/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": ms,
            "steps": steps,
            "inputs": "valid logits rows (one copy per sequence) and every small array, "
                      "from pinned host memory",
            "results": "loss statistics, per-token logp and entropy; dlogits stays on the "
                       "device for the backward pass",
            "pipeline": "double-buffered: upload of step i+1 beside compute of step i",
            "effective_h2d_GB_per_s": h2d / (ms / 1e3) / 1e9,
            "host_link": link,
            "loss_last_step": st["loss"]}


def host_link(dev, nbytes=1 << 30, reps=3):
    """Host<->device copy rate of this machine, timed in this run: a 1 GiB pinned
    buffer copied each way with CUDA events (best of `reps`)."""
    import torch
    h = torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)
    d = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    out = {}
    for name, dst, src in (("h2d_GB_per_s", d, h), ("d2h_GB_per_s", h, d)):
        best = float("inf")
        for _ in range(reps + 1):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            dst.copy_(src, non_blocking=True)
            e1.record(stream)
            torch.cuda.synchronize(dev)
            best = min(best, e0.elapsed_time(e1))
        out[name] = nbytes / (best / 1e3) / 1e9
    out["how"] = f"{nbytes >> 20} MiB pinned copy each way, best of {reps} after one warm-up"
    del h, d
    return out


# ----------------------------------------------------------------------------- CPU oracle
def sample_rows(w, n):
    """n rows spread evenly over the batch (keeps the batch's valid fraction)."""
    return np.unique(np.linspace(0, w.R - 1, max(1, n)).round().astype(np.int64))


def _storage(t):
    import torch
    if t.dtype in (torch.bfloat16, torch.float16):
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def sample_logits(w, rows, dev_logits=None):
    """Host copy (element storage) of the given rows of the workload's logits."""
    import torch
    from ppo_policy_loss_gb300 import synth

    if dev_logits is not None:
        t = dev_logits.index_select(0, torch.from_numpy(rows).to(dev_logits.device)).cpu()
    else:
        device = "cuda" if torch.cuda.is_available() else "cpu"
        parts = []
        for b in np.unique(rows // synth.ROW_BLOCK):
            blk = synth.logits_block(w, int(b), device)
            sel = rows[(rows // synth.ROW_BLOCK) == b] - b * synth.ROW_BLOCK
            parts.append(blk[torch.from_numpy(sel).to(blk.device)].cpu())
        t = torch.cat(parts)
    return _storage(t)


def cpu_sample(w, rows, dev_logits=None):
    """Oracle inputs for the sampled rows; logp_old / ref composed from the
    oracle's own logp plus the workload's noise (input preparation)."""
    import oracle
    from ppo_policy_loss_gb300 import synth

    small = synth.small_inputs(w)
    host = sample_logits(w, rows, dev_logits)
    mask, ids = small["mask"][rows], small["ids"][rows]
    _, logp, _ = oracle.row_stats(host, w.dtype, w.V, ids, mask)
    lo = np.where(mask != 0, logp + small["noise_old"][rows], 0.0).astype(np.float32)
    rf = np.where(mask != 0, logp + small["noise_ref"][rows], 0.0).astype(np.float32)
    return dict(host=host, mask=mask, ids=ids, small=small, rows=rows, lo=lo, rf=rf)


def oracle_step(w, s, threads):
    """One oracle pass of the whole step over the sample: the batch's
    advantages, then loss, statistics and the gradient of every sample row."""
    import oracle

    sm = s["small"]
    if w.advantage == "gae":
        A, _ = oracle.gae(sm["rewards"], sm["values"], sm["lengths"], w.gamma, w.lam)
        arow = A.reshape(-1)[s["rows"]]
    else:
        arow = np.repeat(oracle.group_advantages(sm["rewards"], w.group), w.T)[s["rows"]]
    return oracle.policy_loss(s["host"], w.dtype, w.V, s["ids"], s["mask"], arow,
                              logp_old=s["lo"], ref_logp=s["rf"] if w.beta != 0 else None,
                              eps=w.eps, beta=w.beta, c_ent=w.c_ent, grad_scale=1.0,
                              threads=threads)


def _sample_text(w, s, threads, extra=""):
    n, nv = s["rows"].size, int(s["mask"].sum())
    return (f"{n} rows spread evenly over the {w.R}-row batch ({nv} valid, V={w.V} {w.dtype})"
            f"{extra}; fp64 C oracle on {threads} host threads")


def cpu_baseline(w, dev_logits=None, budget_s=15.0, n_rows=512, threads=None):
    """The oracle as it stands, timed on the host cores over a bounded sample
    (all of the process's host threads unless ``threads`` is given)."""
    import oracle

    threads = threads or oracle.default_threads()
    s = cpu_sample(w, sample_rows(w, n_rows), dev_logits)
    t0 = time.time()
    done = 0
    while True:
        oracle_step(w, s, threads)
        done += s["rows"].size
        if time.time() - t0 >= budget_s:
            break
    dt = time.time() - t0
    return {"value": done / dt, "unit": "tokens/s", "cores": threads, "kind": "oracle",
            "sample": _sample_text(w, s, threads, f", repeated for {dt:.1f} s")}


def cpu_baselines(w, name, dev_logits=None, budget_s=15.0):
    """The oracle on the host cores in two settings, all host threads and one
    thread, for the timed workload (its all-thread figure is the line's
    cpu_baseline) and, on smaller samples, for every other workload."""
    from ppo_policy_loss_gb300 import synth

    out = cpu_baseline(w, dev_logits, budget_s=0.4 * budget_s)
    out["one_thread"] = cpu_baseline(w, dev_logits, budget_s=0.15 * budget_s, n_rows=64, threads=1)
    per = {}
    others = [n for n in OTHER_WORKLOADS + (WORKLOAD,) if n != name]
    for other in others:
        wk = synth.WORKLOADS[other]
        b = 0.45 * budget_s / (2 * len(others))
        per[other] = {"all_threads": cpu_baseline(wk, None, budget_s=b, n_rows=64),
                      "one_thread": cpu_baseline(wk, None, budget_s=b, n_rows=16, threads=1)}
    out["other_workloads"] = per
    return out


def run_reference(args):
    """The reference arm: the fp64 CPU oracle, each step a bounded sample."""
    world, rank, _ = dist_env()
    if rank != 0:
        return
    import oracle

    w = workload_for(args)
    threads = oracle.default_threads()
    # size each step so that warm-up + timed steps take about args.ref_seconds
    probe = cpu_sample(w, sample_rows(w, 64))
    t0 = time.time()
    oracle_step(w, probe, threads)
    per_row = (time.time() - t0) / probe["rows"].size
    n = int(args.ref_seconds / (args.steps + args.warmup) / max(per_row, 1e-9))
    s = cpu_sample(w, sample_rows(w, min(max(n, 16), 4096)))
    for _ in range(args.warmup):
        oracle_step(w, s, threads)
    t0 = time.time()
    for _ in range(args.steps):
        oracle_step(w, s, threads)
    dt = time.time() - t0
    value = args.steps * s["rows"].size / dt
    out = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
           "data": "synthetic", "impl": "reference",
           "config": {"workload": f"{args.workload}: {DESCRIBE.get(args.workload, '')}",
                      "B": w.B, "T": w.T, "V": w.V, "step_sample_rows": int(s["rows"].size)},
           "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                            "sample": "each step: " + _sample_text(w, s, threads)},
           "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


# ----------------------------------------------------------------------------- LM-head leg
def lmhead_config(R, D, V):
    rows = "32 seqs x T=1024" if R == LMHEAD_SHAPE["R"] else "profiling slice"
    name = {1024: "qwen3_0p6b_lmhead", 2048: "qwen3_1p7b_lmhead", 2560: "qwen3_4b_lmhead",
            4096: "qwen3_8b_lmhead"}.get(D, f"lmhead_d{D}")
    return {"workload": f"{name}: {R} rows ({rows}) x D={D} hidden -> "
                        f"V={V} bf16 LM head, hidden ~N(0,1), W ~N(0, 9/D), ids uniform",
            "rows": R, "D": D, "V": V,
            "l2": f"weight {V * D * 2 / 1e9:.2f} GB > 129 MB L2, swept every launch; no flush"}


def lmhead_inputs_dev(dev, rows=0, dim=0):
    import torch
    c = LMHEAD_SHAPE
    D = dim or c["D"]
    g = torch.Generator(device=dev).manual_seed(c["seed"])
    h = torch.randn((rows or c["R"], D), generator=g, device=dev).to(torch.bfloat16)
    w = (torch.randn((c["V"], D), generator=g, device=dev)
         * (c["logit_sd"] / D ** 0.5)).to(torch.bfloat16)
    ids = torch.randint(0, c["V"], (h.shape[0],), generator=g, device=dev)
    return h, w, ids


def lmhead_cpu(h, w, ids, budget_s, n_rows=64):
    """The oracle (fp64 matmul, then row statistics) on a sample of rows."""
    import oracle
    rows = np.unique(np.linspace(0, h.shape[0] - 1, n_rows).round().astype(np.int64))
    hs, ws_, idn = _storage(h[rows].cpu()), _storage(w.cpu()), ids.cpu().numpy()[rows]
    threads = oracle.default_threads()
    t0, done = time.time(), 0
    while True:
        oracle.lmhead_row_stats(hs, ws_, idn, "bf16", threads)
        done += rows.size
        if time.time() - t0 >= budget_s:
            break
    dt = time.time() - t0
    return {"value": done / dt, "unit": "rows/s", "cores": threads, "kind": "oracle",
            "sample": (f"{rows.size} rows spread over the {h.shape[0]}-row batch, full V={w.shape[0]}, "
                       f"D={w.shape[1]}; numpy fp64 matmul + C row statistics, repeated for "
                       f"{dt:.1f} s")}


def run_lmhead(args):
    import torch

    import ppo_policy_loss_gb300 as rl

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    rl.build()
    rl.load()
    h, w, ids = lmhead_inputs_dev(dev, args.lmhead_rows, args.lmhead_dim)
    R, D = h.shape
    V = w.shape[0]
    logp = torch.empty(R, device=dev)
    ent = torch.empty(R, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    ws = torch.zeros(max(16, rl.rl_lmhead_workspace_size(R, V)), dtype=torch.uint8, device=dev)
    n_sl, grid, group, _ = rl.rl_lmhead_plan(R, D, V, ws.numel())
    stream = torch.cuda.current_stream(dev)

    def launch(hh, out_lp, out_en):
        rl.rl_lmhead_logprobs(hh, D, w, D, "bf16", R, D, V, ids, out_lp, out_en, None, status, ws,
                              ws.numel(), stream)

    for _ in range(args.warmup):
        launch(h, logp, ent)
    torch.cuda.synchronize(dev)
    assert int(status.item()) == 0

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize(dev)

    kev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    sampler = ClockSampler(int(vis.split(",")[local]) if vis else local)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    sampler.start()
    time.sleep(0.3)
    t0.record(stream)
    for i in range(args.steps):
        kev[i][0].record(stream)
        launch(h, logp, ent)
        kev[i][1].record(stream)
    t1.record(stream)
    barrier()
    clocks = sampler.stop()
    ms_step = max_over_ranks(t0.elapsed_time(t1), dev) / args.steps
    kern_ms = statistics.mean(a.elapsed_time(b) for a, b in kev)
    flops = 2.0 * R * D * V
    peak, peak_kind = bf16_peak()
    achieved = flops / (kern_ms / 1e3) / 1e12

    # end to end: hidden states and ids uploaded from pinned host memory, the
    # log-probs and entropies read back, every step (the weight stays resident)
    e2e = None
    if args.e2e_steps > 0:
        hh = torch.empty(h.shape, dtype=h.dtype, pin_memory=True)
        hh.copy_(h)
        hid = torch.empty(ids.shape, dtype=ids.dtype, pin_memory=True)
        hid.copy_(ids)
        o_lp = torch.empty(R, pin_memory=True)
        o_en = torch.empty(R, pin_memory=True)
        dh, dids = torch.empty_like(h), torch.empty_like(ids)
        steps = max(1, min(args.steps, args.e2e_steps))
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            dh.copy_(hh, non_blocking=True)
            dids.copy_(hid, non_blocking=True)
            rl.rl_lmhead_logprobs(dh, D, w, D, "bf16", R, D, V, dids, logp, ent, None, status, ws,
                                  ws.numel(), stream)
            o_lp.copy_(logp, non_blocking=True)
            o_en.copy_(ent, non_blocking=True)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        ms = max_over_ranks(e0.elapsed_time(e1), dev) / steps
        e2e = {"value": world * R / (ms / 1e3), "unit": "rows/s",
               "h2d_bytes_per_step": R * D * 2 + R * 8, "d2h_bytes_per_step": 2 * R * 4,
               "ms_per_step": ms, "steps": steps,
               "note": "LM-head weight resident on the device (model state)"}
    out = {
        "metric": LMHEAD_METRIC, "value": world * R / (ms_step / 1e3), "unit": "rows/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded)", "config": dict(lmhead_config(R, D, V),
                                                    parallelism="replicas" if world > 1 else "single GPU",
                                                    split={"vocab_slices": n_sl, "ctas": grid,
                                                           "row_tiles_per_group": group}),
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak, "peak_source": peak_kind,
                     # no full-size record: the weight's sweeps through L2 depend on the
                     # row count, so a slice's traffic does not scale by rows (see profiles/)
                     "traffic": None,
                     "alg_flops_per_launch": flops, "kernel": "rl_lmhead_logprobs",
                     "kernel_ms": kern_ms},
        "e2e": e2e, "gpu_launches": args.steps, "clocks": clocks,
    }
    sust = bf16_sustained_peak()
    if sust:  # back-to-back launches run under the power cap: the sustained figure beside the burst one
        out["roofline"]["peak_sustained"] = sust
        out["roofline"]["frac_of_sustained"] = achieved / sust
    if rank == 0 and not args.no_cpu_baseline:
        out["cpu_baseline"] = lmhead_cpu(h, w, ids, args.cpu_seconds)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(out), flush=True)


LMHEAD_TRAIN_METRIC = ("policy loss + gradients from hidden states through the LM head, rows/s "
                       "(Qwen3 head, V=151936 bf16); % of tensor roofline")


def run_lmhead_train(args):
    """The training op from hidden states (lmhead_train.lmhead_policy_loss): the
    forward row statistics, the loss launch, then per chunk the recomputed
    gradient dz, dhidden and dweight, all on this library's kernels, on the
    Qwen3-0.6B head over the GRPO workload's 32 x 1024 rows (its mask, ids and
    rewards).  Four R x D x V products per step; each kernel is also timed
    alone for its own roofline."""
    import torch

    import ppo_policy_loss_gb300 as rl
    from ppo_policy_loss_gb300 import lmhead_train, synth, torch_api

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    rl.build()
    rl.load()
    h, W, _ = lmhead_inputs_dev(dev, args.lmhead_rows, args.lmhead_dim)
    R, D = h.shape
    V = W.shape[0]
    wl = synth.WORKLOADS[WORKLOAD]
    T = wl.T
    B = R // T
    small = synth.small_inputs(wl)
    t = lambda x: torch.from_numpy(np.ascontiguousarray(x)).to(dev)
    ids, mask = t(small["ids"][:R] % V), t(small["mask"][:R])
    rewards = t(small["rewards"][:B])
    opts = dict(eps=wl.eps, beta=0.0, c_ent=0.01, grad_scale=1.0)
    if B % wl.group == 0:  # whole groups: the loss launch normalises the rewards itself
        opts["group_size"] = wl.group
    stream = torch.cuda.current_stream(dev)

    def step():
        return lmhead_train.lmhead_policy_loss(h, W, ids, mask, rewards, B, T, **opts)

    for _ in range(args.warmup):
        out = step()
    torch.cuda.synchronize(dev)
    assert int(out["status"].item()) == 0 and torch_api.read_stats(out["loss_stats"])["device_error"] == 0
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    sampler = ClockSampler(int(vis.split(",")[local]) if vis else local)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler.start()
    time.sleep(0.3)
    t0.record(stream)
    for _ in range(args.steps):
        out = step()
    t1.record(stream)
    torch.cuda.synchronize(dev)
    clocks = sampler.stop()
    ms_step = t0.elapsed_time(t1) / args.steps
    del out
    torch.cuda.empty_cache()

    # each kernel alone, back to back (CUDA events around 5 launches after 3)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    parts = torch.empty((R, 4), device=dev)
    nb = rl.rl_lmhead_workspace_size(R, V)
    ws = torch.zeros(max(nb, 16), dtype=torch.uint8, device=dev)
    rl.rl_lmhead_row_partials(h, D, W, D, "bf16", R, D, V, ids, parts, status, ws, nb)
    coef = torch_api.policy_loss_from_partials(parts, "bf16", V, ids, mask, rewards, B, T,
                                               **opts)["row_coef"]
    dz = torch.empty((R, V), dtype=torch.bfloat16, device=dev)
    dH = torch.empty_like(h)
    dW = torch.empty((V, D), dtype=torch.float32, device=dev)
    kernels = {
        "rl_lmhead_row_partials": lambda: rl.rl_lmhead_row_partials(h, D, W, D, "bf16", R, D, V, ids,
                                                                    parts, status, ws, nb),
        "rl_lmhead_dlogits": lambda: rl.rl_lmhead_dlogits(h, D, W, D, "bf16", R, D, V, ids, coef, dz, V,
                                                          status),
        "rl_lmhead_dhidden": lambda: rl.rl_lmhead_dhidden(dz, V, W, D, "bf16", R, D, V, dH, D, status),
        "rl_lmhead_dweight": lambda: rl.rl_lmhead_dweight(dz, V, h, D, "bf16", R, D, V, dW, D, 0, status),
    }
    flops = 2.0 * R * D * V
    peak, peak_kind = bf16_peak()
    sust = bf16_sustained_peak()
    per = {}
    for name, fn in kernels.items():
        for _ in range(3):
            fn()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(5):
            fn()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        ms = e0.elapsed_time(e1) / 5
        tf = flops / (ms / 1e3) / 1e12
        per[name] = {"ms": ms, "TFLOP_per_s": tf, "frac_of_burst": tf / peak,
                     "frac_of_sustained": (tf / sust) if sust else None}
    assert int(status.item()) == 0
    achieved = 4 * flops / (ms_step / 1e3) / 1e12
    top = max(per, key=lambda k: per[k]["ms"])
    out = {
        "metric": LMHEAD_TRAIN_METRIC, "value": R / (ms_step / 1e3), "unit": "rows/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded)",
        "config": dict(lmhead_config(R, D, V), loss="GRPO group rewards in the loss launch, c_ent=0.01",
                       valid_tokens=int(small["mask"][:R].sum()), parallelism="single GPU"),
        "roofline": {"bound": "tensor", "achieved": achieved,
                     "peak": sust if sust else peak, "unit": "TFLOP/s",
                     "frac": achieved / (sust if sust else peak),
                     "peak_source": "measured (sustained: four GEMMs back to back)" if sust else peak_kind,
                     "peak_burst": peak, "frac_of_burst": achieved / peak, "traffic": None,
                     "alg_flops_per_step": 4 * flops, "dominant_kernel": top},
        "kernels": per, "e2e": None, "clocks": clocks,
        # per step: statistics, loss, and dlogits / dhidden / dweight per chunk of sequences
        "gpu_launches": args.steps * (2 + 3 * -(-B // lmhead_train._seqs_per_chunk(B, T, V, 2, 16 << 30))),
    }
    if rank == 0:
        print(json.dumps(out), flush=True)


def run_lmhead_reference(args):
    """Reference arm of the LM-head leg: the oracle on host cores, bounded sample."""
    world, rank, _ = dist_env()
    if rank != 0:
        return
    import torch
    c = LMHEAD_SHAPE
    h, w, ids = lmhead_inputs_dev(torch.device("cpu"))
    n = 16   # rows per step: each pass also decodes the whole weight to fp64
    base = lmhead_cpu(h, w, ids, 0.0, n)
    for _ in range(args.warmup - 1):
        lmhead_cpu(h, w, ids, 0.0, n)
    t0 = time.time()
    for _ in range(args.steps):
        lmhead_cpu(h, w, ids, 0.0, n)
    dt = time.time() - t0
    value = args.steps * n / dt
    print(json.dumps({
        "metric": LMHEAD_METRIC, "value": value, "unit": "rows/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "impl": "reference",
        "config": dict(lmhead_config(c["R"], c["D"], c["V"]), step_sample_rows=n),
        "cpu_baseline": {"value": value, "unit": "rows/s", "cores": base["cores"],
                         "kind": "oracle", "sample": "each step: " + base["sample"]},
        "e2e": {"value": value, "unit": "rows/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0}}), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--workload", default=WORKLOAD,
                    choices=["tiny_grpo", "qwen3_0p6b_grpo", "long_seq_grpo", "ppo_gae",
                             "large_grpo"])
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--ref-seconds", type=float, default=120.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip timing the other workloads after the headline")
    ap.add_argument("--no-aux", action="store_true",
                    help="skip timing the O(B*T) kernels beside the loss")
    ap.add_argument("--global-token-mean", action="store_true",
                    help="with N > 1: normalise by the token count summed over ranks")
    ap.add_argument("--seqs", type=int, default=0,
                    help="profiling only: keep the first SEQS sequences")
    ap.add_argument("--vocab", type=int, default=0, help="profiling only: another V")
    ap.add_argument("--dtype", choices=["f32", "bf16", "f16"], default=None,
                    help="profiling only: another logits dtype")
    ap.add_argument("--seq-len", type=int, default=0, help="profiling only: another T")
    ap.add_argument("--all-valid", action="store_true",
                    help="profiling only: every position valid (no masked rows)")
    ap.add_argument("--c-ent", type=float, default=None,
                    help="profiling only: another entropy coefficient (0 drops the entropy term)")
    ap.add_argument("--lmhead", action="store_true",
                    help="time rl_lmhead_logprobs on the Qwen3-0.6B LM head instead")
    ap.add_argument("--lmhead-train", action="store_true",
                    help="time the policy loss and its gradients from hidden states through the "
                         "Qwen3-0.6B LM head (rl_lmhead_* kernels) instead")
    ap.add_argument("--lmhead-rows", type=int, default=0,
                    help="profiling only: rows of the LM-head leg (default 32768)")
    ap.add_argument("--lmhead-dim", type=int, default=0,
                    help="hidden size of the LM-head leg (default 1024, Qwen3-0.6B; "
                         "2048, 2560, 4096 are the Qwen3-1.7B/4B/8B heads)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.lmhead_train:
        if args.impl == "reference":
            print(json.dumps({"impl": "reference", "unavailable": "the LM-head training leg has no CPU "
                              "reference arm; run the default leg"}))
        else:
            run_lmhead_train(args)
    elif args.lmhead:
        (run_lmhead_reference if args.impl == "reference" else run_lmhead)(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
