"""Guard regions around every output and workspace (a stand-in for a memory
checker): each output is a slice of a larger buffer whose 4 KiB before and
after hold a canary bit pattern, and is itself pre-filled with NaN; each
workspace is followed by 4 KiB of canary bytes.  After a call through the C
ABI the canaries must be intact (no store past either end of an output or
past the workspace size the library reported) and no NaN may survive in an
output (every element written).

The shapes reach the places where an out-of-bounds store could hide: ragged
last TMA boxes (T not a multiple of the stage), partial head or channel
groups of a warp, ragged last chunks of the time-chunked path, the
few-lane long-sequence Givens path that forms A in its workspace, and the
delta rule's ragged last 64-step chunk."""
import math

import pytest
import torch

from scan_linear_recurrences_gb300 import _binding as b
from scan_linear_recurrences_gb300 import inputs
from scan_linear_recurrences_gb300.build import build

pytestmark = pytest.mark.gpu

GUARD = 1024                 # floats on each side (4 KiB)
CANARY = 0x5A5AC3A5          # int32 pattern of the output guards
WS_CANARY = 0xA7             # byte pattern after each workspace


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    build()
    b.lib()
    yield
    b.mgs_check()


class Guarded:
    """An fp32 output of `shape` inside a buffer with canary guards, pre-filled with NaN."""

    def __init__(self, name, shape):
        self.name = name
        self.n = math.prod(shape)
        self.buf = torch.full((GUARD + self.n + GUARD,), CANARY, dtype=torch.int32, device="cuda")
        self.t = self.buf[GUARD:GUARD + self.n].view(torch.float32).view(shape)
        self.t.fill_(float("nan"))

    def check(self):
        head, tail = self.buf[:GUARD], self.buf[GUARD + self.n:]
        assert bool((head == CANARY).all()), f"{self.name}: store before the start of the output"
        assert bool((tail == CANARY).all()), f"{self.name}: store past the end of the output"
        assert not bool(torch.isnan(self.t).any()), f"{self.name}: elements left unwritten"


class GuardedWs:
    """A workspace of the size the library asks for, followed by canary bytes."""

    def __init__(self, op, B, T, HD, k):
        self.n = b.mgs_workspace_size(op, B, T, HD, k)
        self.buf = torch.full((self.n + 4 * GUARD,), WS_CANARY, dtype=torch.uint8, device="cuda")
        self.ptr = self.buf if self.n else None

    def check(self, what):
        assert bool((self.buf[self.n:] == WS_CANARY).all()), f"{what}: store past the workspace size"


def _run(outs, wss, what):
    b.mgs_check()
    for o in outs:
        o.check()
    for w in wss:
        w.check(what)


def _cuda(d):
    return {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in d.items()}


# ---------------------------------------------------------------- matrix_affine_scan (+ recompute backward)
@pytest.mark.parametrize("B,T,H,k", [
    (3, 37, 5, 8),      # ragged stage, partial head group
    (2, 45, 3, 4), (2, 33, 3, 16), (2, 81, 12, 1),
    (1, 333, 3, 8),     # time-chunked, ragged last chunk
    (1, 1000, 3, 16),
])
def test_guard_matrix_affine_scan(B, T, H, k):
    d = _cuda(inputs.mas_inputs(B, T, H, k, seed=31 + T, h0="normal"))
    h = Guarded("h", (B, T, H, k))
    wf = GuardedWs(b.MGS_OP_MATRIX_AFFINE_SCAN_FWD, B, T, H, k)
    b.mgs_matrix_affine_scan_fwd(d["A"], d["b"], d["h0"], h.t, B, T, H, k, wf.ptr, wf.n)
    _run([h], [wf], "mas fwd")
    dA, db, dh0 = Guarded("dA", (B, T, H, k, k)), Guarded("db", (B, T, H, k)), Guarded("dh0", (B, H, k))
    wb = GuardedWs(b.MGS_OP_MATRIX_AFFINE_SCAN_BWD, B, T, H, k)
    b.mgs_matrix_affine_scan_bwd(d["A"], d["h0"], h.t, d["grad_h"], dA.t, db.t, dh0.t, B, T, H, k, wb.ptr, wb.n)
    _run([dA, db, dh0], [wb], "mas bwd")
    rA, rb, r0 = Guarded("dA rc", (B, T, H, k, k)), Guarded("db rc", (B, T, H, k)), Guarded("dh0 rc", (B, H, k))
    wr = GuardedWs(b.MGS_OP_MATRIX_AFFINE_SCAN_BWD_RECOMPUTE, B, T, H, k)
    b.mgs_matrix_affine_scan_bwd_recompute(d["A"], d["b"], d["h0"], d["grad_h"], rA.t, rb.t, r0.t, B, T, H, k,
                                           wr.ptr, wr.n)
    _run([rA, rb, r0], [wr], "mas bwd recompute")


# ---------------------------------------------------------------- matrix_scan (+ no-allocation forward)
@pytest.mark.parametrize("B,T,H,k", [
    (2, 13, 5, 8), (2, 21, 3, 4), (2, 17, 3, 16), (2, 30, 8, 1),
    (1, 333, 2, 8),     # time-chunked, ragged last chunk
    (1, 515, 3, 16),
])
def test_guard_matrix_scan(B, T, H, k):
    d = _cuda(inputs.ms_inputs(B, T, H, k, seed=41 + T))
    P = Guarded("P", (B, T, H, k, k))
    wf = GuardedWs(b.MGS_OP_MATRIX_SCAN_FWD, B, T, H, k)
    b.mgs_matrix_scan_fwd(d["A"], P.t, B, T, H, k, wf.ptr, wf.n)
    _run([P], [wf], "ms fwd")
    dA = Guarded("dA", (B, T, H, k, k))
    wb = GuardedWs(b.MGS_OP_MATRIX_SCAN_BWD, B, T, H, k)
    b.mgs_matrix_scan_bwd(d["A"], P.t, d["grad_P"], dA.t, B, T, H, k, wb.ptr, wb.n)
    _run([dA], [wb], "ms bwd")
    Pn = Guarded("P noalloc", (B, T, H, k, k))
    b.mgs_matrix_scan_fwd_noalloc(d["A"], Pn.t, B, T, H, k)
    _run([Pn], [], "ms fwd noalloc")


# ---------------------------------------------------------------- parallel_scan_log (saved h and recompute)
@pytest.mark.parametrize("B,T,D", [(3, 50, 132), (5, 33, 36), (2, 257, 1024), (2, 17, 8),
                                   # several blocks a warp; 2048 channel groups (one warp per 128 channels)
                                   (2, 1500, 36), (64, 20, 1024),
                                   # 40 blocks a warp: the recompute backward's 80 KB of dynamic shared memory
                                   (1, 20000, 12)])
def test_guard_parallel_scan_log(B, T, D):
    d = _cuda(inputs.psl_inputs(B, T, D, seed=51 + T + D, with_h0=True))
    h, lh = Guarded("h", (B, T, D)), Guarded("log_h", (B, T, D))
    b.mgs_parallel_scan_log_fwd(d["log_coeffs"], d["log_values"], d["log_h0"], h.t, lh.t, B, T, D)
    _run([h, lh], [], "psl fwd")
    dlc, dlv, dl0 = Guarded("dlc", (B, T, D)), Guarded("dlv", (B, T, D)), Guarded("dl0", (B, D))
    b.mgs_parallel_scan_log_bwd(d["log_coeffs"], d["log_values"], d["log_h0"], h.t, d["grad_h"], dlc.t, dlv.t,
                                dl0.t, B, T, D)
    _run([dlc, dlv, dl0], [], "psl bwd")
    qlc, qlv, ql0 = Guarded("dlc rc", (B, T, D)), Guarded("dlv rc", (B, T, D)), Guarded("dl0 rc", (B, D))
    wr = GuardedWs(b.MGS_OP_PARALLEL_SCAN_LOG_BWD, B, T, D, 0)
    b.mgs_parallel_scan_log_bwd(d["log_coeffs"], d["log_values"], d["log_h0"], None, d["grad_h"], qlc.t, qlv.t,
                                ql0.t, B, T, D, wr.ptr, wr.n)
    _run([qlc, qlv, ql0], [wr], "psl bwd recompute")


# ---------------------------------------------------------------- linear_scan
@pytest.mark.parametrize("B,T,D", [(3, 77, 132), (1, 2000, 32), (2, 45, 4), (64, 30, 1024), (1, 20000, 12),
                                   (1, 33000, 4)])
def test_guard_linear_scan(B, T, D):
    d = _cuda(inputs.linear_inputs(B, T, D, seed=61 + T + D))
    h = Guarded("h", (B, T, D))
    wf = GuardedWs(b.MGS_OP_LINEAR_SCAN_FWD, B, T, D, 1)
    b.mgs_linear_scan_fwd(d["a"], d["b"], d["h0"], h.t, B, T, D, wf.ptr, wf.n)
    _run([h], [wf], "linear fwd")
    da, db, dh0 = Guarded("da", (B, T, D)), Guarded("db", (B, T, D)), Guarded("dh0", (B, D))
    wb = GuardedWs(b.MGS_OP_LINEAR_SCAN_BWD, B, T, D, 1)
    b.mgs_linear_scan_bwd(d["a"], d["h0"], h.t, d["grad_h"], da.t, db.t, dh0.t, B, T, D, wb.ptr, wb.n)
    _run([da, db, dh0], [wb], "linear bwd")


# ---------------------------------------------------------------- Givens-mesh scans
@pytest.mark.parametrize("B,T,H,with_a", [
    (3, 130, 5, False),   # one lane per block, ragged stage, no gate
    (5, 33, 100, True),   # partial head group
    (40, 9, 256, True),   # eight lanes per block, a block shorter than a stage
    (2, 300, 3, True),    # few lanes, long sequence: the workspace path
    (1, 517, 4, False),
])
def test_guard_givens_affine_scan(B, T, H, with_a):
    d = _cuda(inputs.givens_affine_inputs(B, T, H, 8, seed=71 + T, h0="normal", with_a=with_a))
    a = d["a"]
    h = Guarded("h", (B, T, H, 8))
    wf = GuardedWs(b.MGS_OP_GIVENS_AFFINE_SCAN_FWD, B, T, H, 8)
    b.mgs_givens_affine_scan_fwd(d["theta"], a, d["b"], d["h0"], h.t, B, T, H, 8, wf.ptr, wf.n)
    _run([h], [wf], "givens affine fwd")
    dth, dbv, dh0 = Guarded("d_theta", (B, T, H, 28)), Guarded("db", (B, T, H, 8)), Guarded("dh0", (B, H, 8))
    outs = [dth, dbv, dh0]
    da = None
    if with_a:
        da = Guarded("da", (B, T, H, 8))
        outs.append(da)
    wb = GuardedWs(b.MGS_OP_GIVENS_AFFINE_SCAN_BWD, B, T, H, 8)
    b.mgs_givens_affine_scan_bwd(d["theta"], a, d["h0"], h.t, d["grad_h"], dth.t, da.t if da else None, dbv.t,
                                 dh0.t, B, T, H, 8, wb.ptr, wb.n)
    _run(outs, [wb], "givens affine bwd")


@pytest.mark.parametrize("B,T,H", [(3, 33, 9), (2, 50, 3), (2, 300, 4), (1, 517, 5)])
def test_guard_givens_matrix_scan(B, T, H):
    d = _cuda(inputs.givens_matrix_inputs(B, T, H, 8, seed=81 + T))
    P = Guarded("P", (B, T, H, 8, 8))
    wf = GuardedWs(b.MGS_OP_GIVENS_MATRIX_SCAN_FWD, B, T, H, 8)
    b.mgs_givens_matrix_scan_fwd(d["theta"], P.t, B, T, H, 8, wf.ptr, wf.n)
    _run([P], [wf], "givens matrix fwd")
    dth = Guarded("d_theta", (B, T, H, 28))
    wb = GuardedWs(b.MGS_OP_GIVENS_MATRIX_SCAN_BWD, B, T, H, 8)
    b.mgs_givens_matrix_scan_bwd(d["theta"], P.t, d["grad_P"], dth.t, B, T, H, 8, wb.ptr, wb.n)
    _run([dth], [wb], "givens matrix bwd")


# ---------------------------------------------------------------- delta rule
@pytest.mark.parametrize("B,T,H", [(2, 100, 3), (1, 64, 1), (2, 130, 2), (3, 7, 2)])
def test_guard_delta_rule(B, T, H):
    d = _cuda(inputs.delta_inputs(B, T, H, 64, seed=91 + T, with_S0=True))
    o, ST = Guarded("o", (B, T, H, 64)), Guarded("S_T", (B, H, 64, 64))
    w = GuardedWs(b.MGS_OP_DELTA_SCAN_FWD, B, T, H, 64)
    b.mgs_delta_scan_fwd(d["q"], d["k"], d["v"], d["beta"], d["S0"], o.t, ST.t, B, T, H, 64, w.ptr, w.n)
    _run([o, ST], [w], "delta fwd")
