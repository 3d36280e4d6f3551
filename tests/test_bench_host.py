"""Host logic of bench.py for more than one rank, on CPU with gloo.

The timed GPU path runs one process per GPU with no data-path collective;
what the ranks share is a barrier and the max over ranks of the step time,
and, for ``--impl reference``, the rule that rank 0 alone runs the oracle
and prints.  These tests run that logic as world-size-2 gloo process groups.
"""
from __future__ import annotations

import json
import os
import socket
import subprocess
import sys

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


class _Args:
    impl = "reference"   # gloo even where a GPU is present


def _rank_main(rank: int, world: int, port: int, q) -> None:
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist
    w, r, local = bench.dist_setup(_Args())
    # each rank's step time differs; every rank must see the slowest one
    slowest = bench.max_over_ranks(1.25 + r, w)
    bench.barrier(w)
    q.put((r, w, local, slowest, dist.get_backend()))
    dist.destroy_process_group()


def test_max_over_ranks_and_barrier_gloo():
    ctx = torch.multiprocessing.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    try:
        got = sorted(q.get(timeout=120) for _ in procs)
    finally:
        for p in procs:
            p.join(timeout=60)
    assert [g[0] for g in got] == [0, 1]
    for rank, world, local, slowest, backend in got:
        assert world == 2 and local == rank
        assert slowest == 2.25
        assert backend == "gloo"
    assert all(p.exitcode == 0 for p in procs)


def test_single_rank_needs_no_process_group():
    assert bench.max_over_ranks(3.5, 1) == 3.5
    bench.barrier(1)   # a no-op without a process group


def test_reference_arm_under_torchrun_prints_once():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py",
           "--impl", "reference", "--gpus", "2", "--steps", "2", "--warmup", "3",
           "--workload", "tiny_f32", "--ref-seconds", "2"]
    env = dict(os.environ, OMP_NUM_THREADS="2")
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    assert d["n_gpus"] == 2 and d["steps"] == 2 and d["warmup"] == 3
    assert d["higher_is_better"] is True and d["unit"] == "tokens/s" and d["value"] > 0
    assert d["config"]["workload"] == "tiny_f32"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-GPU refusal")
def test_our_arm_refuses_to_run_without_a_gpu():
    r = subprocess.run([sys.executable, "bench.py", "--steps", "1", "--warmup", "3"], cwd=ROOT,
                       capture_output=True, text=True, timeout=300)
    assert r.returncode != 0
    assert "no CUDA device" in r.stderr


def test_source_hash_ignores_comments_and_layout_only():
    """A DRAM traffic record is keyed by a hash of the kernel's code: editing
    a comment or re-indenting keeps it, any change of code (string literals
    included) drops it."""
    base = 'int f(int a) {\n    return a + 1;  // one\n}\nconst char *s = "a // b";\n'
    same = ('/* doc */ int f(int a)\n{\n  return a + 1;   /* one */\n}\n'
            'const char *s = "a // b";   // trailing\n')
    assert bench.code_tokens(base) == bench.code_tokens(same)
    for changed in (base.replace("+ 1", "+ 2"), base.replace('"a // b"', '"a //  b"'),
                    base.replace("return a", "return  -a")):
        assert bench.code_tokens(changed) != bench.code_tokens(base)
    # every kernel that has a record hashes to a fixed-length hex string
    for stage in bench.KERNEL_SOURCES:
        h = bench.kernel_source_hash(stage)
        assert len(h) == 16 and int(h, 16) >= 0


def test_roofline_work_of_each_workload():
    """The roofline's numerators: compulsory HBM bytes (x, B, C, dt, A, D and
    the initial state read; y and the final state written) and flops (per
    token and head 2NP chunk state + 2NP output from the state + (Q + 1)P on
    the causal half of the intra-chunk product + 2NP/Q state pass, per token
    and group (Q + 1)N for C B^T), worked out by hand for each workload."""
    from state_space_model_gb300 import inputs as gen
    # 2.7B layer: x = y = 8*4096*80*64*2 B = 335,544,320; B + C = 2*8*4096*128*2 =
    # 16,777,216; dt = 8*4096*80*4 = 10,485,760; A + D = 640; final = 8*80*64*128*4
    # = 20,971,520
    expect_bytes = {"mamba2_2p7b": 2 * 335_544_320 + 16_777_216 + 10_485_760 + 640
                    + 20_971_520}
    b, f = bench.path_work(gen.WORKLOADS["mamba2_2p7b"])
    assert b == expect_bytes["mamba2_2p7b"] == 719_323_776
    T, H, P, N, Q, G = 8 * 4096, 80, 64, 128, 256, 1
    assert f == T * H * (4 * N * P + (Q + 1) * P + 2 * N * P / Q) + T * G * (Q + 1) * N
    # rounded figures of the other workloads (MB, GFLOP)
    for name, mb, gf in [("tiny_f32", 0.172, 0.00239), ("mamba2_130m", 58.46, 9.96),
                         ("hybrid_g8", 620.8, 88.47), ("long_64k", 2256.5, 417.7)]:
        b, f = bench.path_work(gen.WORKLOADS[name])
        assert abs(b / 1e6 - mb) / mb < 1e-3 and abs(f / 1e9 - gf) / gf < 1e-3, name
