"""Benchmark of the scan primitives on one GB300 (or N replicas under torchrun).

One step = forward + backward of every scan primitive at its benchmark shape:
  matrix_affine_scan lab      B=128 T=64   H=8  k=8
  matrix_scan long-T Givens   B=16  T=1024 H=8  k=8
  parallel_scan_log minGRU    B=64  T=4096 D=1024
  matrix_affine_scan scaled   B=32  T=8192 H=64 k=8
Inputs are seeded synthetic tensors resident in HBM; the two small shapes fit in
L2, so L2 is flushed (a 512 MiB write) before each of their calls.  Each call is
bracketed by CUDA events on the launching stream; the step's device time is the
sum of its eight calls.  value = algorithmic bytes of a step / that time (GB/s).

Prints one JSON line.  ``--impl reference`` times the float64 CPU oracle on the
host cores instead (bounded sample of the same workloads).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "fwd+bwd scan µs and achieved HBM GB/s (% of peak) per op and shape"
WORKLOAD_IDS = (1, 2, 3, 4)
FALLBACK_HBM_GBS = 6800.0
FLUSH_BYTES = 512 << 20


# ---------------------------------------------------------------- algorithmic bytes
def op_bytes(w, direction):
    """Bytes each argument contributes when read or written once (fp32)."""
    B, T, H, k = w.B, w.T, w.H, w.k
    if w.op == "mas":
        steps = B * T * H
        init = B * H * k * 4
        if direction == "fwd":  # read A, b; write h; read h0
            return steps * 4 * (k * k + 2 * k) + (init if w.h0 != "none" else 0)
        # read A, grad_h, h; write dA, db; read h0 (if any); write dh0
        return steps * 4 * (2 * k * k + 3 * k) + (init if w.h0 != "none" else 0) + init
    if w.op == "ms":
        steps = B * T * H
        return steps * 4 * (2 * k * k if direction == "fwd" else 4 * k * k)
    if w.op == "lin":
        elems = B * T * H  # H holds D
        init = B * H * 4
        if direction == "fwd":  # read a, b; write h; read h0
            return elems * 12 + (init if w.h0 != "none" else 0)
        # read a, grad_h, h; write da, db; read h0, write dh0
        return elems * 20 + (init if w.h0 != "none" else 0) + init
    if w.op == "gas":  # angles N = k(k-1)/2 per step instead of the k x k matrix
        steps, n = B * T * H, k * (k - 1) // 2
        init = B * H * k * 4
        if direction == "fwd":  # read theta, a, b; write h; read h0
            return steps * 4 * (n + 3 * k) + (init if w.h0 != "none" else 0)
        # read theta, a, grad_h, h; write d_theta, da, db; read h0, write dh0
        return steps * 4 * (2 * n + 5 * k) + (init if w.h0 != "none" else 0) + init
    if w.op == "delta":  # forward only: read q, k, v, beta, S0; write o, S_T (k holds D)
        elems, state = B * T * H * k, B * H * k * k
        return (4 * elems + B * T * H + 2 * state) * 4 if direction == "fwd" else 0
    if w.op == "gms":
        steps, n = B * T * H, k * (k - 1) // 2
        if direction == "fwd":  # read theta; write P
            return steps * 4 * (n + k * k)
        return steps * 4 * (2 * n + 2 * k * k)  # read theta, P, grad_P; write d_theta
    elems = B * T * H  # H holds D for parallel_scan_log
    init = B * H * 4
    if direction == "fwd":  # read lc, lv; write h; read log_h0
        return elems * 12 + init
    return elems * 24 + 2 * init  # read lc, lv, g, h; write dlc, dlv; read log_h0, write d_log_h0


def measured_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


# sources each kernel family is built from (a change to any of them makes
# recorded ncu counters stale; mgs_launch.h holds only host declarations)
KERNEL_SOURCES = {"mas": ["mgs_mas.cu"], "ms": ["mgs_ms.cu"], "psl": ["mgs_psl.cu"],
                  "gas": ["mgs_givens.cu"], "gms": ["mgs_givens.cu"]}
COMMON_SOURCES = ["mgs_device.cuh", "mgs_tiles.cuh"]
CHUNK_SOURCES = {"ms": ["mgs_chunk.cuh"], "mas": ["mgs_chunk.cuh"], "psl": [], "gas": [], "gms": []}
TRAFFIC_JSON = os.path.join(ROOT, "profiles", "traffic.json")


def kernel_source_hash(op):
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "scan_linear_recurrences_gb300", "csrc")
    for f in KERNEL_SOURCES[op] + CHUNK_SOURCES[op] + COMMON_SOURCES:
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def committed_traffic(op, key):
    """DRAM bytes per launch of kernel `key` from the committed ncu record, only
    if it was taken on the current sources of that kernel family."""
    try:
        with open(TRAFFIC_JSON) as f:
            d = json.load(f)
    except Exception:
        return None
    e = d.get("kernels", {}).get(key)
    if e is None or e.get("source_hash") != kernel_source_hash(op):
        return None
    return e.get("dram_bytes_per_launch")


def record_traffic(csv_path, rows, workloads):
    """Turns an ncu CSV (dram__bytes_read/write.sum per launch, taken with
    --batch-rows `rows`) into profiles/traffic.json, scaling each kernel's
    bytes to a full launch by the batch rows processed."""
    import csv
    from scan_linear_recurrences_gb300 import inputs
    with open(csv_path) as f:
        table = list(csv.reader(f))
    hi = next(i for i, r in enumerate(table) if "Kernel Name" in r)
    hdr = table[hi]
    ki, mi, vi = hdr.index("Kernel Name"), hdr.index("Metric Name"), hdr.index("Metric Value")
    by_op = {inputs.WORKLOADS[i].op: inputs.WORKLOADS[i] for i in workloads}
    acc = {}
    for r in table[hi + 1:]:
        if r[mi] not in ("dram__bytes_read.sum", "dram__bytes_write.sum"):
            continue
        name = r[ki].split("(")[0].split("::")[-1].split("<")[0].strip()
        op = name.split("_")[0]
        w = by_op[op]
        key = f"{name}@c{w.cid}"
        acc.setdefault(key, {"op": op, "w": w, "read": [], "write": []})
        acc[key]["read" if "read" in r[mi] else "write"].append(float(r[vi].replace(",", "")))
    out = {"how": f"ncu --metrics dram__bytes_read.sum,dram__bytes_write.sum on --batch-rows {rows}, "
                  "scaled to the full batch; writes still dirty in L2 at kernel end are not counted",
           "kernels": {}}
    for key, a in acc.items():
        w = a["w"]
        scale = w.B / min(w.B, rows)
        rd, wr = statistics.mean(a["read"]), statistics.mean(a["write"])
        out["kernels"][key] = {"dram_bytes_per_launch": round((rd + wr) * scale),
                               "read_bytes": round(rd * scale), "write_bytes": round(wr * scale),
                               "source_hash": kernel_source_hash(a["op"]), "scale": scale}
    with open(TRAFFIC_JSON, "w") as f:
        json.dump(out, f, indent=1)
    return out


# ---------------------------------------------------------------- clocks
class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


# ---------------------------------------------------------------- multi-rank aggregation
def max_over_ranks(x, world, device="cpu"):
    """Largest value of x across the ranks (the slowest rank sets the time)."""
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_gbps(step_bytes_per_rank, world, ms_step_max):
    """Weak scaling: every rank processes its own copy of the step's work, so
    the job moves world * step_bytes in the slowest rank's step time."""
    return step_bytes_per_rank * world / (ms_step_max * 1e-3) / 1e9


# ---------------------------------------------------------------- GPU arm
def givens_peak_memory(torch, api, device, B=128, T=64, H=8, k=8):
    """Peak device memory of one forward+backward through the Givens affine
    scan at the pages' memory-benchmark shape (B=128, T=64, d=64, k=8): the
    angle-fused op against the generic path that first builds A = G(theta)
    diag(a) with eager autograd ops and then runs matrix_affine_scan.  Memory
    held before the call (the inputs) is not counted."""
    from scan_linear_recurrences_gb300 import inputs

    d = inputs.givens_affine_inputs(B, T, H, k, seed=BASE_SEED_GIVENS_MEMORY, device=device, h0="normal")
    g = d["grad_h"]

    def mesh_eager(theta):
        M = torch.eye(k, device=device).expand(B, T, H, k, k)
        n = 0
        for layer in range(k):
            for p in range(layer % 2, k - 1, 2):
                c, s = torch.cos(theta[..., n, None]), torch.sin(theta[..., n, None])
                x, y = M[..., p, :], M[..., p + 1, :]
                rows = list(M.unbind(-2))
                rows[p], rows[p + 1] = c * x - s * y, s * x + c * y
                M = torch.stack(rows, dim=-2)
                n += 1
        return M

    def run(fused):
        leaves = {n: d[n].clone().requires_grad_(True) for n in ("theta", "a", "b", "h0")}
        torch.cuda.synchronize()
        torch.cuda.reset_peak_memory_stats(device)
        base = torch.cuda.memory_allocated(device)
        if fused:
            h = api.givens_affine_scan(leaves["theta"], leaves["a"], leaves["b"], leaves["h0"])
        else:
            A = mesh_eager(leaves["theta"]) * leaves["a"].unsqueeze(-2)
            h = api.matrix_affine_scan(A, leaves["b"], leaves["h0"])
        (h * g).sum().backward()
        torch.cuda.synchronize()
        return (torch.cuda.max_memory_allocated(device) - base) / 1e6

    return {"shape": f"B={B} T={T} H={H} k={k} (d={H * k})", "angle_fused_MB": round(run(True), 2),
            "eager_mesh_then_matrix_affine_scan_MB": round(run(False), 2)}


BASE_SEED_GIVENS_MEMORY = 20261202 + 99


def copy_floor_us(torch, flush, stream, nbytes, reps):
    """Median microseconds of a plain device copy moving `nbytes` (half read,
    half written), timed as the L2-resident shapes' calls are: L2 flushed,
    then CUDA events around the one call.  The floor those calls' times sit
    on: launch, the first HBM round trip and the bytes."""
    src = torch.empty(max(1, nbytes // 8), dtype=torch.float32, device=flush.device)
    dst = torch.empty_like(src)
    evs = []
    for i in range(reps + 3):
        flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        dst.copy_(src)
        e1.record(stream)
        if i >= 3:
            evs.append((e0, e1))
    torch.cuda.synchronize()
    return round(statistics.median(x.elapsed_time(y) for x, y in evs) * 1e3, 2)


def delta_flops(w, C=64):
    """Floating-point operations of the chunked WY forward per call: per
    64-step chunk the products K K^T, Q K^T, the forward substitution for
    [W | U], W S^T, Q S^T, tril(Q K^T) U' and U'^T K, i.e. 4 C^2 D + 3 C D^2
    multiply-adds (2 flops each); chunks are counted whole."""
    D = w.k
    chunks = -(-w.T // C)
    return 2 * (4 * C * C * D + 3 * C * D * D) * chunks * w.B * w.H


def fp32_fma_peak_tflops():
    """fp32 peak of the CUDA cores from unit counts and clock: SMs x 128 FMA
    lanes x 2 flops x the maximum SM clock (MEASURED_PEAKS.json sm_max_mhz,
    else the nominal 2070 MHz)."""
    import torch
    mhz = 2070.0
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            mhz = float(json.load(f).get("sm_max_mhz", mhz))
    except Exception:
        pass
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    return sms * 128 * 2 * mhz * 1e6 / 1e12


class Runner:
    """Holds one workload's device buffers and runs its fwd / bwd calls."""

    def kernels_per_step(self):
        """Kernel launches of one fwd + one bwd call: the time-chunked
        matrix_affine_scan and matrix_scan paths (a nonzero workspace) run
        three launches a call, every other step workload one."""
        per_call = 3 if self.w.op in ("mas", "ms") and self.nf > 0 else 1
        return 2 * per_call

    def __init__(self, w, torch, b, api, device):
        self.w = w
        self.t = torch
        self.api = api
        self.device = device
        d = w.make(device=device)
        self.inp = d
        B, T, H, k = w.B, w.T, w.H, w.k
        e = lambda *s: torch.empty(s, dtype=torch.float32, device=device)
        if w.op == "mas":
            self.h = e(B, T, H, k)
            self.dA, self.db, self.dh0 = e(B, T, H, k, k), e(B, T, H, k), e(B, H, k)
            self.ws_f, self.nf = api.workspace(b.MGS_OP_MATRIX_AFFINE_SCAN_FWD, B, T, H, k, device)
            self.ws_b, self.nb = api.workspace(b.MGS_OP_MATRIX_AFFINE_SCAN_BWD, B, T, H, k, device)
        elif w.op == "lin":
            self.h = e(B, T, H)
            self.da, self.db, self.dh0 = e(B, T, H), e(B, T, H), e(B, H)
            self.ws_f, self.nf = api.workspace(b.MGS_OP_LINEAR_SCAN_FWD, B, T, H, 1, device)
            self.ws_b, self.nb = api.workspace(b.MGS_OP_LINEAR_SCAN_BWD, B, T, H, 1, device)
        elif w.op == "ms":
            self.P, self.dA = e(B, T, H, k, k), e(B, T, H, k, k)
            self.ws_f, self.nf = api.workspace(b.MGS_OP_MATRIX_SCAN_FWD, B, T, H, k, device)
            self.ws_b, self.nb = api.workspace(b.MGS_OP_MATRIX_SCAN_BWD, B, T, H, k, device)
        elif w.op == "gas":
            self.h = e(B, T, H, k)
            self.dth, self.da, self.db, self.dh0 = e(B, T, H, k * (k - 1) // 2), e(B, T, H, k), e(B, T, H, k), e(B, H, k)
            self.ws_f, self.nf = api.workspace(b.MGS_OP_GIVENS_AFFINE_SCAN_FWD, B, T, H, k, device)
            self.ws_b, self.nb = api.workspace(b.MGS_OP_GIVENS_AFFINE_SCAN_BWD, B, T, H, k, device)
        elif w.op == "gms":
            self.P, self.dth = e(B, T, H, k, k), e(B, T, H, k * (k - 1) // 2)
            self.ws_f, self.nf = api.workspace(b.MGS_OP_GIVENS_MATRIX_SCAN_FWD, B, T, H, k, device)
            self.ws_b, self.nb = api.workspace(b.MGS_OP_GIVENS_MATRIX_SCAN_BWD, B, T, H, k, device)
        elif w.op == "delta":
            self.o, self.ST = e(B, T, H, k), e(B, H, k, k)
            self.ws_f, self.nf = api.workspace(b.MGS_OP_DELTA_SCAN_FWD, B, T, H, k, device)
        else:
            self.h = e(B, T, H)
            self.dlc, self.dlv, self.dl0 = e(B, T, H), e(B, T, H), e(B, H)
        self.b = b

    def part(self, r0, r1):
        """A view of this runner restricted to batch rows [r0, r1) (contiguous
        slices: the batch dimension is outermost in every tensor)."""
        v = object.__new__(Runner)
        v.__dict__.update(self.__dict__)
        from dataclasses import replace
        v.w = replace(self.w, B=r1 - r0)
        v.inp = {k: (t[r0:r1] if t is not None else None) for k, t in self.inp.items()}
        for name in ("h", "dA", "db", "dh0", "P", "dlc", "dlv", "dl0", "da"):
            if hasattr(self, name):
                setattr(v, name, getattr(self, name)[r0:r1])
        return v

    def fwd(self, stream):
        w, d, b = self.w, self.inp, self.b
        if w.op == "mas":
            b.mgs_matrix_affine_scan_fwd(d["A"], d["b"], d["h0"], self.h, w.B, w.T, w.H, w.k, self.ws_f, self.nf, stream)
        elif w.op == "lin":
            b.mgs_linear_scan_fwd(d["a"], d["b"], d["h0"], self.h, w.B, w.T, w.H, self.ws_f, self.nf, stream)
        elif w.op == "ms":
            b.mgs_matrix_scan_fwd(d["A"], self.P, w.B, w.T, w.H, w.k, self.ws_f, self.nf, stream)
        elif w.op == "gas":
            b.mgs_givens_affine_scan_fwd(d["theta"], d["a"], d["b"], d["h0"], self.h, w.B, w.T, w.H, w.k,
                                         self.ws_f, self.nf, stream)
        elif w.op == "gms":
            b.mgs_givens_matrix_scan_fwd(d["theta"], self.P, w.B, w.T, w.H, w.k, self.ws_f, self.nf, stream)
        elif w.op == "delta":
            b.mgs_delta_scan_fwd(d["q"], d["k"], d["v"], d["beta"], d["S0"], self.o, self.ST, w.B, w.T, w.H, w.k,
                                 self.ws_f, self.nf, stream)
        else:
            b.mgs_parallel_scan_log_fwd(d["log_coeffs"], d["log_values"], d["log_h0"], self.h, None,
                                        w.B, w.T, w.H, None, 0, stream)

    def bwd(self, stream):
        w, d, b = self.w, self.inp, self.b
        if w.op == "mas":
            b.mgs_matrix_affine_scan_bwd(d["A"], d["h0"], self.h, d["grad_h"], self.dA, self.db, self.dh0,
                                         w.B, w.T, w.H, w.k, self.ws_b, self.nb, stream)
        elif w.op == "lin":
            b.mgs_linear_scan_bwd(d["a"], d["h0"], self.h, d["grad_h"], self.da, self.db, self.dh0,
                                  w.B, w.T, w.H, self.ws_b, self.nb, stream)
        elif w.op == "ms":
            b.mgs_matrix_scan_bwd(d["A"], self.P, d["grad_P"], self.dA, w.B, w.T, w.H, w.k, self.ws_b, self.nb, stream)
        elif w.op == "gas":
            b.mgs_givens_affine_scan_bwd(d["theta"], d["a"], d["h0"], self.h, d["grad_h"], self.dth, self.da,
                                         self.db, self.dh0, w.B, w.T, w.H, w.k, self.ws_b, self.nb, stream)
        elif w.op == "gms":
            b.mgs_givens_matrix_scan_bwd(d["theta"], self.P, d["grad_P"], self.dth, w.B, w.T, w.H, w.k, self.ws_b,
                                         self.nb, stream)
        elif w.op == "delta":
            pass  # forward only (the pages' DeltaMinGRU row is its chunked-WY forward)
        else:
            b.mgs_parallel_scan_log_bwd(d["log_coeffs"], d["log_values"], d["log_h0"], self.h, d["grad_h"],
                                        self.dlc, self.dlv, self.dl0, w.B, w.T, w.H, None, 0, stream)

    # e2e: host buffers in pinned memory, copies inside the timed region
    def host_setup(self, parts):
        t, b, api = self.t, self.b, self.api
        self.host_in = {k: v.cpu().pin_memory() for k, v in self.inp.items() if v is not None}
        outs = self.outputs()
        self.host_out = [t.empty(o.shape, dtype=o.dtype, pin_memory=True) for o in outs]
        self.h2d = sum(v.numel() * 4 for v in self.host_in.values())
        self.d2h = sum(o.numel() * 4 for o in outs)
        rows = self.w.B // parts
        self.parts = []
        for i in range(parts):
            r0, r1 = i * rows, (self.w.B if i == parts - 1 else (i + 1) * rows)
            v = self.part(r0, r1)
            v.host_in = {k: h[r0:r1] for k, h in self.host_in.items()}
            v.host_out = [h[r0:r1] for h in self.host_out]
            # a part may take a different (chunked) plan than the full batch
            w = v.w
            op_ids = {"mas": (b.MGS_OP_MATRIX_AFFINE_SCAN_FWD, b.MGS_OP_MATRIX_AFFINE_SCAN_BWD),
                      "ms": (b.MGS_OP_MATRIX_SCAN_FWD, b.MGS_OP_MATRIX_SCAN_BWD),
                      "lin": (b.MGS_OP_LINEAR_SCAN_FWD, b.MGS_OP_LINEAR_SCAN_BWD)}.get(w.op)
            if op_ids:
                v.ws_f, v.nf = api.workspace(op_ids[0], w.B, w.T, w.H, w.k, self.device)
                v.ws_b, v.nb = api.workspace(op_ids[1], w.B, w.T, w.H, w.k, self.device)
            self.parts.append(v)

    def outputs(self):
        if self.w.op == "mas":
            return [self.h, self.dA, self.db, self.dh0]
        if self.w.op == "ms":
            return [self.P, self.dA]
        if self.w.op == "lin":
            return [self.h, self.da, self.db, self.dh0]
        return [self.h, self.dlc, self.dlv, self.dl0]

    def e2e_issue(self, s_in, s_comp, s_out, ev):
        """One end-to-end pass of this workload on three streams: host->device
        copies of the inputs (s_in), fwd+bwd through the C ABI (s_comp),
        device->host copies of the results (s_out).  Events order each buffer's
        reuse across passes, so transfers of one workload overlap the compute of
        another and the two copy directions run at the same time."""
        t = self.t
        s_in.wait_event(ev["comp"])      # previous pass has consumed the inputs
        with t.cuda.stream(s_in):
            for k, v in self.host_in.items():
                self.inp[k].copy_(v, non_blocking=True)
        ev["in"].record(s_in)
        s_comp.wait_event(ev["in"])
        s_comp.wait_event(ev["out"])     # previous pass has read the outputs
        self.fwd(s_comp.cuda_stream)
        self.bwd(s_comp.cuda_stream)
        ev["comp"].record(s_comp)
        s_out.wait_event(ev["comp"])
        with t.cuda.stream(s_out):
            for dst, src in zip(self.host_out, self.outputs()):
                dst.copy_(src, non_blocking=True)
        ev["out"].record(s_out)


def run_gpu(args):
    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    device = f"cuda:{local}"

    from scan_linear_recurrences_gb300 import _binding as b
    from scan_linear_recurrences_gb300 import api, inputs
    from scan_linear_recurrences_gb300.build import build
    build()
    b.lib()

    ids = [int(x) for x in args.workloads.split(",")]
    # the report-only shapes may be named too (profiling their kernels alone)
    ws = [inputs.WORKLOADS[i] if i in inputs.WORKLOADS else inputs.EXTRA_WORKLOADS[i] for i in ids]
    if args.batch_rows:
        # profiling only: a smaller case of the same kernels (fewer batch rows)
        from dataclasses import replace
        ws = [replace(w, B=min(w.B, args.batch_rows)) for w in ws]
    runners = [Runner(w, torch, b, api, device) for w in ws]
    small = {r.w.cid: r.w.B * r.w.T * r.w.H * r.w.k * r.w.k * 4 * 3 < (256 << 20) for r in runners}
    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=device)
    stream = torch.cuda.current_stream()
    sid = stream.cuda_stream

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    def one_step(evs):
        for r in runners:
            if small[r.w.cid]:
                flush.zero_()
            e0, e1, e2 = evs[r.w.cid]
            e0.record(stream)
            r.fwd(sid)
            e1.record(stream)
            r.bwd(sid)
            e2.record(stream)

    for _ in range(args.warmup):
        one_step({r.w.cid: [torch.cuda.Event(enable_timing=True) for _ in range(3)] for r in runners})
    b.mgs_check(sid)

    sampler = ClockSampler(local) if rank == 0 else None
    if sampler:
        sampler.start()
        time.sleep(0.3)
    all_evs = []
    barrier()
    t_wall = time.perf_counter()
    for _ in range(args.steps):
        evs = {r.w.cid: [torch.cuda.Event(enable_timing=True) for _ in range(3)] for r in runners}
        one_step(evs)
        all_evs.append(evs)
    barrier()
    wall = time.perf_counter() - t_wall
    clocks = sampler.stop() if sampler else None
    b.mgs_check(sid)

    # per-op times (ms)
    per = {}
    for r in runners:
        f = [ev[r.w.cid][0].elapsed_time(ev[r.w.cid][1]) for ev in all_evs]
        bw = [ev[r.w.cid][1].elapsed_time(ev[r.w.cid][2]) for ev in all_evs]
        per[r.w.cid] = (f, bw)
    step_ms = [sum(per[c][0][i] + per[c][1][i] for c in per) for i in range(args.steps)]
    ms_step = max_over_ranks(statistics.mean(step_ms), world, device)

    peak, peak_kind = measured_peak()
    step_bytes = sum(op_bytes(r.w, "fwd") + op_bytes(r.w, "bwd") for r in runners)
    value = whole_job_gbps(step_bytes, world, ms_step)

    ops = {}
    dominant = None
    for r in runners:
        w = r.w
        f, bw = per[w.cid]
        fm, bm = statistics.median(f), statistics.median(bw)
        fb, bb_ = op_bytes(w, "fwd"), op_bytes(w, "bwd")
        key = f"{w.op}_c{w.cid}"
        ops[key] = {
            "shape": w.name, "fwd_us": round(fm * 1e3, 2), "bwd_us": round(bm * 1e3, 2),
            "fwd_bwd_us": round((fm + bm) * 1e3, 2),
            "fwd_GBps": round(fb / (fm * 1e-3) / 1e9, 1), "bwd_GBps": round(bb_ / (bm * 1e-3) / 1e9, 1),
            "fwd_bwd_GBps": round((fb + bb_) / ((fm + bm) * 1e-3) / 1e9, 1),
            "fwd_bwd_pct_of_peak": round(100 * (fb + bb_) / ((fm + bm) * 1e-3) / 1e9 / peak, 1),
            "l2": "flushed" if small[w.cid] else "inputs larger than L2",
        }
        if small[w.cid]:
            # a plain copy of the same bytes, timed the same way (not part of the step)
            ops[key]["same_bytes_copy_us"] = [copy_floor_us(torch, flush, stream, fb, args.steps),
                                              copy_floor_us(torch, flush, stream, bb_, args.steps)]
        for direction, tms, nbytes in (("fwd", statistics.mean(f), fb), ("bwd", statistics.mean(bw), bb_)):
            if dominant is None or tms > dominant[1]:
                dominant = (f"{w.op}_{direction}_c{w.cid}", tms, nbytes, w, direction)

    kname, kms, kbytes, kw, kdir = dominant
    achieved = kbytes / (kms * 1e-3) / 1e9
    chunked = kw.op in ("ms", "mas") and b.mgs_workspace_size(
        b.MGS_OP_MATRIX_SCAN_FWD if kw.op == "ms" else b.MGS_OP_MATRIX_AFFINE_SCAN_FWD, kw.B, kw.T, kw.H, kw.k) > 0
    # the time-chunked path is three launches: aggregates, carry chain, outputs
    kernel_symbol = (f"{kw.op}_{kdir}_agg_kernel+chain_kernel+{kw.op}_{kdir}_out_kernel" if chunked
                     else f"{kw.op}_{kdir}_kernel")
    if kw.op == "delta":
        kernel_symbol = "delta_wy_kernel+delta_state_kernel"
    traffic = committed_traffic(kw.op, f"{kernel_symbol}@c{kw.cid}")
    roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4), "traffic": traffic,
                "kernel": kernel_symbol, "workload": kw.name,
                "algorithmic_bytes_per_launch": kbytes, "peak_kind": f"{peak_kind} hbm_gbs (copy, burst)"}

    # e2e through the C ABI with pinned host buffers; copies inside the timed region
    e2e = None
    if not args.no_e2e:
        # the two large workloads stream in 16-row parts so their transfers overlap their compute
        for r in runners:
            big = op_bytes(r.w, "fwd") + op_bytes(r.w, "bwd") > (1 << 30)
            r.host_setup(parts=max(1, r.w.B // 16) if big else 1)
        units = [p for r in runners for p in r.parts]
        s_in, s_comp, s_out = (torch.cuda.Stream(device=device) for _ in range(3))
        evs = [{k: torch.cuda.Event() for k in ("in", "comp", "out")} for _ in units]
        for ev in evs:
            for e_ in ev.values():
                e_.record(stream)
        barrier()
        for u, ev in zip(units, evs):  # warm-up pass
            u.e2e_issue(s_in, s_comp, s_out, ev)
        torch.cuda.synchronize()
        barrier()
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ev0.record(s_in)
        s_comp.wait_event(ev0)
        s_out.wait_event(ev0)
        n_e2e = max(1, min(args.steps, 3))
        for _ in range(n_e2e):
            for u, ev in zip(units, evs):
                u.e2e_issue(s_in, s_comp, s_out, ev)
        s_out.wait_stream(s_in)
        s_out.wait_stream(s_comp)
        ev1.record(s_out)
        torch.cuda.synchronize()
        barrier()
        e2e_ms = max_over_ranks(ev0.elapsed_time(ev1) / n_e2e, world, device)
        b.mgs_check(sid)
        e2e = {"value": round(whole_job_gbps(step_bytes, world, e2e_ms), 1), "unit": "GB/s",
               "h2d_bytes_per_step": sum(r.h2d for r in runners), "d2h_bytes_per_step": sum(r.d2h for r in runners),
               "ms_per_step": round(e2e_ms, 3),
               "how": "pinned host buffers; H2D, C-ABI fwd+bwd and D2H on three streams, pipelined over "
                      "16-batch-row parts of the large workloads"}

    extra = {}
    if not args.no_extra:
        for w in inputs.EXTRA_WORKLOADS.values():
            r = Runner(w, torch, b, api, device)
            fs, bs = [], []
            for it in range(args.warmup + 10):
                flush.zero_()
                e0, e1, e2 = (torch.cuda.Event(enable_timing=True) for _ in range(3))
                e0.record(stream)
                r.fwd(sid)
                e1.record(stream)
                r.bwd(sid)
                e2.record(stream)
                torch.cuda.synchronize()
                if it >= args.warmup:
                    fs.append(e0.elapsed_time(e1))
                    bs.append(e1.elapsed_time(e2))
            fm, bm = statistics.median(fs), statistics.median(bs)
            nbytes = op_bytes(w, "fwd") + op_bytes(w, "bwd")
            if w.op == "delta":
                flops = delta_flops(w)
                extra[f"{w.op}_c{w.cid}"] = {
                    "shape": w.name, "fwd_us": round(fm * 1e3, 2), "fwd_GBps": round(nbytes / (fm * 1e-3) / 1e9, 1),
                    "fwd_TFLOPs": round(flops / (fm * 1e-3) / 1e12, 2), "flops_per_call": flops,
                    "pct_of_fp32_fma_peak": round(100 * flops / (fm * 1e-3) / 1e12 / fp32_fma_peak_tflops(), 1),
                    "l2": "flushed"}
                del r
                continue
            extra[f"{w.op}_c{w.cid}"] = {"shape": w.name, "fwd_us": round(fm * 1e3, 2), "bwd_us": round(bm * 1e3, 2),
                                         "fwd_bwd_us": round((fm + bm) * 1e3, 2),
                                         "fwd_bwd_GBps": round(nbytes / ((fm + bm) * 1e-3) / 1e9, 1),
                                         "l2": "flushed"}
            del r
        # parallel_scan_log backward in recompute mode (h not saved) on the
        # minGRU shape and the pages' lab and long-T shapes: DRAM bytes are 28
        # per element on the minGRU shape (log_coeffs and log_values read by
        # both passes, grad_h read, two gradients written), 20 where h is
        # recomputed in registers (few lanes)
        psl_extra = [Runner(w, torch, b, api, device) for w in inputs.EXTRA_WORKLOADS.values() if w.op == "psl"]
        for r in runners + psl_extra:
            w = r.w
            if w.op != "psl":
                continue
            d = r.inp
            ws, nws = api.workspace(b.MGS_OP_PARALLEL_SCAN_LOG_BWD, w.B, w.T, w.H, 0, device)
            ts = []
            for it in range(args.warmup + 10):
                flush.zero_()
                e0, e1 = (torch.cuda.Event(enable_timing=True) for _ in range(2))
                e0.record(stream)
                b.mgs_parallel_scan_log_bwd(d["log_coeffs"], d["log_values"], d["log_h0"], None, d["grad_h"],
                                            r.dlc, r.dlv, r.dl0, w.B, w.T, w.H, ws, nws, sid)
                e1.record(stream)
                torch.cuda.synchronize()
                if it >= args.warmup:
                    ts.append(e0.elapsed_time(e1))
            bm = statistics.median(ts)
            # the library's rule for its one-launch diagonal-scan kernels
            in_regs = 1 <= w.T <= 32768 and w.B * ((w.H + 31) // 32) < 2048
            per_elem = 20 if in_regs else 28
            nbytes = w.B * w.T * w.H * per_elem + 2 * w.B * w.H * 4 + (0 if in_regs else 2 * nws)
            extra[f"psl_c{w.cid}_bwd_recompute"] = {
                "shape": w.name, "bwd_us": round(bm * 1e3, 2), "workspace_bytes": nws,
                "GBps": round(nbytes / (bm * 1e-3) / 1e9, 1),
                "bytes": f"{per_elem} per element" + ("" if in_regs else " + checkpoints"), "l2": "flushed"}
            del ws
        del psl_extra
        # matrix_affine_scan backward in recompute mode (h not saved) on the
        # scaled shape: per step A and b read by both passes, grad_h read,
        # dA and db written (4 (2k^2 + 2k + k + k^2 + k) = 896 bytes at k = 8),
        # plus h0 read, dh0 written and the checkpoints written and read
        for r in runners:
            w = r.w
            if w.op != "mas" or w.cid != 4:
                continue
            d = r.inp
            ws, nws = api.workspace(b.MGS_OP_MATRIX_AFFINE_SCAN_BWD_RECOMPUTE, w.B, w.T, w.H, w.k, device)
            ts = []
            for it in range(args.warmup + 10):
                e0, e1 = (torch.cuda.Event(enable_timing=True) for _ in range(2))
                e0.record(stream)
                b.mgs_matrix_affine_scan_bwd_recompute(d["A"], d["b"], d["h0"], d["grad_h"], r.dA, r.db, r.dh0,
                                                       w.B, w.T, w.H, w.k, ws, nws, sid)
                e1.record(stream)
                torch.cuda.synchronize()
                if it >= args.warmup:
                    ts.append(e0.elapsed_time(e1))
            bm = statistics.median(ts)
            k = w.k
            nbytes = w.B * w.T * w.H * 4 * (3 * k * k + 4 * k) + 2 * w.B * w.H * k * 4 + 2 * nws
            extra[f"mas_c{w.cid}_bwd_recompute"] = {
                "shape": w.name, "bwd_us": round(bm * 1e3, 2), "workspace_bytes": nws,
                "GBps": round(nbytes / (bm * 1e-3) / 1e9, 1), "pct_of_peak": round(100 * nbytes / (bm * 1e-3) / 1e9 /
                                                                                   measured_peak()[0], 1),
                "bytes": f"{4 * (3 * k * k + 4 * k)} per step + checkpoints", "l2": "inputs larger than L2"}
            del ws
        b.mgs_check(sid)
        # the pages' memory shape, and the long-sequence shape (time-chunked, still from the angles)
        extra["givens_peak_memory"] = givens_peak_memory(torch, api, device)
        extra["givens_peak_memory_long_T"] = givens_peak_memory(torch, api, device, B=16, T=1024)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        cpu = cpu_baseline(runners, min_s=args.cpu_seconds)

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms_step, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": " + ".join(r.w.name for r in runners) + ", fwd+bwd each",
                       "l2": "flushed before the two L2-resident shapes; the others exceed L2",
                       "step_bytes": step_bytes, "wall_s_timed_region": round(wall, 4)},
            # the report-only shapes first and the per-op lines of the step
            # last, so that a reader keeping only the end of the line keeps them
            "extra_ops_not_in_step": extra, "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": args.steps * sum(r.kernels_per_step() for r in runners), "clocks": clocks,
            "impl": "libmgscan", "ops": ops,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


# ---------------------------------------------------------------- CPU (oracle) legs
def _oracle_sample(w, rows, device_inputs=None):
    """Float64 oracle inputs for `rows` batch rows of workload w."""
    import torch
    d = device_inputs if device_inputs is not None else w.make(device="cpu")
    return {k: (v[:rows].cpu() if isinstance(v, torch.Tensor) else v) for k, v in d.items()}


def _time_oracle(w, s):
    import numpy as np
    import oracle
    f64 = lambda x: None if x is None else np.ascontiguousarray(x.double().numpy())
    if w.op == "mas":
        A, bb, h0, g = f64(s["A"]), f64(s["b"]), f64(s["h0"]), f64(s["grad_h"])
        t0 = time.perf_counter(); oracle.mas_fwd(A, bb, h0); t1 = time.perf_counter()
        oracle.mas_bwd(A, bb, h0 if h0 is not None else np.zeros((A.shape[0], w.H, w.k)), g)
        t2 = time.perf_counter()
    elif w.op == "ms":
        A, G = f64(s["A"]), f64(s["grad_P"])
        t0 = time.perf_counter(); oracle.ms_fwd(A); t1 = time.perf_counter()
        oracle.ms_bwd(A, G); t2 = time.perf_counter()
    else:
        lc, lv, l0, g = f64(s["log_coeffs"]), f64(s["log_values"]), f64(s["log_h0"]), f64(s["grad_h"])
        t0 = time.perf_counter(); oracle.psl_fwd(lc, lv, l0); t1 = time.perf_counter()
        oracle.psl_bwd(lc, lv, l0, g); t2 = time.perf_counter()
    return t2 - t0


def _sample_rows(w, budget_rows):
    return max(1, min(w.B, budget_rows.get(w.cid, w.B)))


# batch rows of each workload one CPU pass processes; passes repeat until the
# CPU leg has run for at least `min_s` seconds (about 10-30 s in total)
CPU_ROWS = {1: 128, 2: 16, 3: 16, 4: 8}


def cpu_baseline(runners, min_s=10.0, rows=None):
    import oracle
    from dataclasses import replace
    rows = rows or CPU_ROWS
    samples = []
    for r in runners:
        w = r.w
        n = _sample_rows(w, rows)
        samples.append((replace(w, B=n), _oracle_sample(w, n, r.inp), w))
    total_b, total_t, passes = 0, 0.0, 0
    while total_t < min_s and passes < 50:
        for ws, s, _ in samples:
            total_t += _time_oracle(ws, s)
            total_b += op_bytes(ws, "fwd") + op_bytes(ws, "bwd")
        passes += 1
    parts = [f"{w.op}_c{w.cid}: {ws.B}/{w.B} batch rows" for ws, _, w in samples]
    return {"value": round(total_b / total_t / 1e9, 3), "unit": "GB/s", "cores": oracle.num_threads(),
            "kind": "oracle",
            "sample": "; ".join(parts) + f"; {passes} passes of fwd+bwd; float64 oracle, OpenMP over lanes",
            "seconds": round(total_t, 2)}


def run_reference(args):
    """The float64 CPU oracle timed as the reference arm (rank 0 only)."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle
    from dataclasses import replace
    from scan_linear_recurrences_gb300 import inputs
    oracle.build()
    ids = [int(x) for x in args.workloads.split(",")]
    ws = [inputs.WORKLOADS[i] for i in ids]
    # each step processes this many batch rows per workload (bounded sample)
    rows = {1: 32, 2: 4, 3: 2, 4: 1}
    samples = []
    for w in ws:
        n = _sample_rows(w, rows)
        wsub = replace(w, B=n)  # same recipe and seed, fewer batch rows
        samples.append((wsub, wsub.make(device="cpu")))
    for _ in range(args.warmup):
        for wsub, s in samples:
            _time_oracle(wsub, s)
    times = []
    for _ in range(args.steps):
        times.append(sum(_time_oracle(wsub, s) for wsub, s in samples))
    step_bytes = sum(op_bytes(wsub, "fwd") + op_bytes(wsub, "bwd") for wsub, _ in samples)
    ms_step = statistics.mean(times) * 1e3
    value = step_bytes / (ms_step * 1e-3) / 1e9
    sample = "; ".join(f"{w.op}_c{w.cid}: {w.B} batch rows" for w, _ in samples)
    line = {
        "metric": METRIC, "value": round(value, 3), "unit": "GB/s", "n_gpus": 0, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": " + ".join(w.name for w in ws) + ", fwd+bwd each (row sample per step)"},
        "impl": "reference",
        "cpu_baseline": {"value": round(value, 3), "unit": "GB/s", "cores": oracle.num_threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 3), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="libmgscan", choices=["libmgscan", "reference"])
    ap.add_argument("--workloads", default=",".join(str(i) for i in WORKLOAD_IDS))
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-extra", action="store_true", help="skip the report-only extra shapes")
    ap.add_argument("--cpu-seconds", type=float, default=10.0, help="minimum CPU-baseline time")
    ap.add_argument("--batch-rows", type=int, default=0,
                    help="profiling: cap every workload's batch rows (smaller case, same kernels)")
    ap.add_argument("--record-traffic", default=None,
                    help="write profiles/traffic.json from this ncu CSV (taken with --batch-rows)")
    args = ap.parse_args()
    if args.record_traffic:
        print(json.dumps(record_traffic(args.record_traffic, args.batch_rows,
                                        [int(x) for x in args.workloads.split(",")]), indent=1))
        return
    if args.warmup < 3 and args.impl != "reference":
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
