"""Host-side logic of bench.py: algorithmic byte counts and the multi-rank
aggregation (max over ranks, whole-job throughput), the latter with two gloo
ranks on the CPU."""
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench
from scan_linear_recurrences_gb300 import inputs


def test_kernel_launch_count_per_step():
    """gpu_launches counts kernels: three a call on the time-chunked paths
    (a nonzero workspace), one otherwise."""
    from types import SimpleNamespace as NS
    k = bench.Runner.kernels_per_step
    assert k(NS(w=NS(op="ms"), nf=4096)) == 6
    assert k(NS(w=NS(op="mas"), nf=4096)) == 6
    assert k(NS(w=NS(op="mas"), nf=0)) == 2
    assert k(NS(w=NS(op="psl"), nf=0)) == 2
    # the step's four workloads: mas lab and scaled single-pass, ms long-T
    # chunked, psl minGRU one launch a call
    from scan_linear_recurrences_gb300 import _binding as b
    plans = [(1, b.MGS_OP_MATRIX_AFFINE_SCAN_FWD), (2, b.MGS_OP_MATRIX_SCAN_FWD), (4, b.MGS_OP_MATRIX_AFFINE_SCAN_FWD)]
    sizes = {cid: b.mgs_workspace_size(op, inputs.WORKLOADS[cid].B, inputs.WORKLOADS[cid].T,
                                       inputs.WORKLOADS[cid].H, inputs.WORKLOADS[cid].k) for cid, op in plans}
    assert sizes[1] == 0 and sizes[4] == 0 and sizes[2] > 0


def test_algorithmic_bytes_per_unit():
    w1, w2, w3, w4 = (inputs.WORKLOADS[i] for i in (1, 2, 3, 4))
    # matrix_affine_scan: 320 B/step forward, 608 B/step backward (+ initial-state terms)
    steps = w1.B * w1.T * w1.H
    assert bench.op_bytes(w1, "fwd") == 320 * steps
    assert bench.op_bytes(w1, "bwd") == 608 * steps + w1.B * w1.H * 8 * 4
    steps4 = w4.B * w4.T * w4.H
    assert bench.op_bytes(w4, "fwd") == 320 * steps4 + w4.B * w4.H * 32
    # matrix_scan: 512 / 1024 B per step
    assert bench.op_bytes(w2, "fwd") == 512 * w2.B * w2.T * w2.H
    assert bench.op_bytes(w2, "bwd") == 1024 * w2.B * w2.T * w2.H
    # parallel_scan_log: 12 / 24 B per element
    n = w3.B * w3.T * w3.H
    assert bench.op_bytes(w3, "fwd") == 12 * n + 4 * w3.B * w3.H
    assert bench.op_bytes(w3, "bwd") == 24 * n + 8 * w3.B * w3.H
    total = sum(bench.op_bytes(w, d) for w in (w1, w2, w3, w4) for d in ("fwd", "bwd"))
    assert total == 25_496_092_672


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    local_ms = [3.0, 5.0][rank]
    m = bench.max_over_ranks(local_ms, world, "cpu")
    q.put((rank, m, bench.whole_job_gbps(1e9, world, m)))
    dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_max_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=100) for _ in procs)
    for p in procs:
        p.join(timeout=30)
        assert p.exitcode == 0
    assert [r[1] for r in res] == [5.0, 5.0]          # slowest rank sets the time
    assert res[0][2] == pytest.approx(2 * 1e9 / 5e-3 / 1e9)  # both ranks' bytes over that time


def test_single_rank_is_identity():
    assert bench.max_over_ranks(4.5, 1) == 4.5


def test_reference_arm_prints_its_line_on_the_cpu():
    """The reference arm (the oracle on the host cores) needs no GPU."""
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "3", "--workloads", "1,2"], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0 and line["unit"] == "GB/s"
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["value"] == line["value"]
