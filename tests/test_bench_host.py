"""Host-side logic of bench.py, including its multi-rank timing reduction run as
two gloo ranks on the CPU (the GPU data path has no cross-rank step)."""
import json
import os
import socket
import subprocess
import sys

import numpy as np
import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402
from ppo_policy_loss_gb300 import synth  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ms = bench.max_over_ranks(10.0 + rank * 2.5, "cpu")
    q.put((rank, ms, bench.whole_job_rate(32768, world, ms)))
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[1] for r in res] == [12.5, 12.5]
    assert res[0][2] == pytest.approx(2 * 32768 / 0.0125)


def test_single_process_identity():
    assert bench.max_over_ranks(3.0, "cpu") == 3.0
    assert bench.whole_job_rate(100, 1, 1000.0) == 100.0


def test_alg_bytes_counts_one_read_of_valid_rows_and_one_write_of_all():
    w = synth.WORKLOADS["qwen3_0p6b_grpo"]
    n_valid = int(synth.small_inputs(w)["mask"].sum())
    b = bench.alg_bytes(w, n_valid)
    assert b == n_valid * w.V * 2 + w.R * w.V * 2 + w.R * 25 + w.B * 4
    assert 15e9 < b < 17e9


def test_sample_rows_spread_and_unique():
    w = synth.WORKLOADS["qwen3_0p6b_grpo"]
    r = bench.sample_rows(w, 512)
    assert r.size == 512 and r[0] == 0 and r[-1] == w.R - 1 and np.all(np.diff(r) > 0)


def test_reference_arm_non_zero_rank_exits_quietly():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--steps", "3", "--warmup", "3"], env=env, capture_output=True,
                         text=True, timeout=120)
    assert out.returncode == 0 and out.stdout.strip() == ""


def test_traffic_record_ignored_when_kernel_changed(tmp_path):
    f = tmp_path / "t.txt"
    f.write_text("kernel_sha: 0000\ndram_bytes_per_launch: 123\n")
    assert bench.recorded_traffic(path=str(f)) is None
    f.write_text(f"kernel_sha: {bench.kernel_sha()}\ndram_bytes_per_launch: 123\n")
    assert bench.recorded_traffic(path=str(f)) == 123.0


def test_kernel_sha_follows_code_not_comments(tmp_path):
    src = tmp_path / "k.cu"
    body = "__global__ void k(int* p) {\n  p[0] = 1;  // one\n}\n"
    src.write_text(body)
    sha = bench.kernel_sha(str(src))
    # comments, trailing blanks and blank lines do not count
    src.write_text("/* a kernel\n   of one store */\n" + body.replace("// one", "// the first element") + "\n\n")
    assert bench.kernel_sha(str(src)) == sha
    # code does
    src.write_text(body.replace("p[0] = 1", "p[0] = 2"))
    assert bench.kernel_sha(str(src)) != sha
    # the default covers the kernel source and the project headers it includes
    assert len(bench.KERNEL_SRCS) == 3 and bench.kernel_sha() == bench.kernel_sha(bench.KERNEL_SRCS)


def test_committed_loss_profiles_name_the_current_kernel():
    """Every traffic record and ncu summary of the loss kernel under profiles/
    was taken on the kernel's current code (the records feed the bench line's
    roofline traffic; a kernel change without new captures fails here)."""
    prof = os.path.join(ROOT, "profiles")
    sha = bench.kernel_sha()
    records = sorted(f for f in os.listdir(prof) if f.startswith("policy_loss_") and f.endswith("_traffic.txt"))
    summaries = sorted(f for f in os.listdir(prof) if f.startswith("policy_loss_") and f.endswith(".md"))
    assert records and summaries
    for f in records:
        name = f[len("policy_loss_"):-len("_traffic.txt")]
        assert bench.recorded_traffic(name) is not None, f
    for f in summaries:
        with open(os.path.join(prof, f)) as fh:
            assert f"kernel_sha {sha}" in fh.read(), f


def test_alg_bytes_ppo_counts_per_token_advantages_and_no_reference():
    w = synth.WORKLOADS["ppo_gae"]
    assert bench.alg_bytes(w, w.R) == 2 * w.R * w.V * 2 + w.R * 21 + w.R * 4


def test_profiling_shape_options_reshape_the_workload():
    import argparse
    base = dict(workload="long_seq_grpo", seqs=0, vocab=0, dtype=None, seq_len=0,
                all_valid=False)
    a = argparse.Namespace(**base)
    assert bench.workload_for(a) == synth.WORKLOADS["long_seq_grpo"] and not bench.reshaped(a)
    b = argparse.Namespace(**dict(base, seqs=8, vocab=50000, dtype="bf16", seq_len=1024,
                                  all_valid=True))
    w = bench.workload_for(b)
    assert (w.B, w.T, w.V, w.dtype, w.lengths) == (8, 1024, 50000, "bf16", ("full",))
    assert bench.reshaped(b)
    mask = synth.small_inputs(w)["mask"]
    assert mask.size == w.R and int(mask.sum()) == w.R  # every position valid


def test_entropy_coefficient_option():
    import argparse
    base = dict(workload="ppo_gae", seqs=0, vocab=0, dtype=None, seq_len=0, all_valid=False,
                c_ent=None)
    assert bench.workload_for(argparse.Namespace(**base)).c_ent == synth.WORKLOADS["ppo_gae"].c_ent
    a = argparse.Namespace(**dict(base, c_ent=0.0))
    w = bench.workload_for(a)
    assert w.c_ent == 0.0 and bench.reshaped(a)  # 0 is a setting, not "unset"
    assert (w.B, w.T, w.V) == (synth.WORKLOADS["ppo_gae"].B, 512, 151936)
