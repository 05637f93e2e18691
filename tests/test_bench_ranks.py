"""The multi-rank host logic of bench.py on CPU (gloo, world size 2): the
max-over-ranks timing, the whole-job throughput, and the reference arm under
torchrun (rank 0 alone reports)."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    mine = [10.0 + 5 * rank, 20.0 - 7 * rank]   # rank 1 slower on the first value only
    got = bench.reduce_max(dist, mine, "cpu")
    out[rank] = got
    dist.destroy_process_group()


def test_reduce_max_over_two_gloo_ranks():
    world, port = 2, _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        assert out[0] == out[1] == [15.0, 20.0]
    # whole-job throughput: every replica's bytes over the slowest replica's time
    assert bench.job_gbps(2, 1e9, 10, 15.0 * 10) == pytest.approx(2 * 1e9 * 10 / 0.15 / 1e9)
    assert bench.reduce_max(None, [1, 2], "cpu") == [1.0, 2.0]


def test_reference_arm_under_torchrun_world_size_two():
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload",
           "decode_q8_ctx4k", "--steps", "1", "--warmup", "3", "--gpus", "2"]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["cpu_baseline"]["kind"] == "oracle"


def test_step_work_accounts_the_fused_append():
    """The one-token decode steps run fused: the roofline kernel then moves the
    appended rows too (fp16 in, encoded row out, both sides); the step's bytes
    are the same either way, and other workloads are unaffected."""
    from attention_quantized_kv_gb300 import workloads as wl
    w = wl.get("append_decode_q4_ctx32k")
    assert bench.fused_decode_step(w)
    b_f, f_f, per_f = bench.step_work(w, True)
    b_u, f_u, per_u = bench.step_work(w, False)
    app = w.n_seqs * w.append_new * w.n_kv * (2 * 256 + 72 + 72)
    assert b_f == b_u and f_f == f_u
    assert per_f[0] - per_u[0] == app
    kv = sum(w.final_lens()) * w.n_kv * (72 + 72)
    assert per_u[0] == kv + 2 * w.n_seqs * w.n_q * 256
    for name in ("decode_q8_ctx4k", "prefill_q8_32k_plus_2k", "decode_16layer_ladder_2x200704"):
        assert not bench.fused_decode_step(wl.get(name))
