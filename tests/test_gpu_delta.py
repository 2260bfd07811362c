"""GPU parity of the delta-rule (DeltaNet) chunked-WY forward against the
float64 oracle: sequences shorter than, equal to and longer than one 64-step
chunk with ragged tails, several heads, with and without an initial state,
the pages' lab and long-T shapes and the throughput shape (sampled rows), and
the degenerate cases."""
import numpy as np
import pytest
import torch

import oracle
from scan_linear_recurrences_gb300 import _binding as b
from scan_linear_recurrences_gb300 import api, inputs
from scan_linear_recurrences_gb300.build import build

from ._parity import assert_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    build()
    b.lib()
    yield
    b.mgs_check()


def _run(d, T, rows=None):
    o, ST = api.delta_scan_fwd(d["q"], d["k"], d["v"], d["beta"], d["S0"], want_state=True)
    b.mgs_check()
    sel = slice(None) if rows is None else rows
    cpu = lambda x: x[sel].cpu() if x is not None else None
    o_ref, ST_ref = oracle.delta_fwd(cpu(d["q"]), cpu(d["k"]), cpu(d["v"]), cpu(d["beta"]), cpu(d["S0"]),
                                     want_state=True)
    assert_close("o", o[sel], o_ref, T)
    assert_close("S_T", ST[sel], ST_ref, T)


@pytest.mark.parametrize("B,T,H,S0", [
    (1, 1, 1, True), (2, 63, 3, True), (2, 64, 2, False), (3, 130, 2, True), (2, 200, 5, False),
    (1, 513, 1, True),
])
def test_delta_shapes(B, T, H, S0):
    d = {k: (v.cuda() if v is not None else None)
         for k, v in inputs.delta_inputs(B, T, H, 64, seed=1300 + B * T + H, with_S0=S0).items()}
    _run(d, T)


@pytest.mark.parametrize("B,T,H", [
    (76, 70, 1),    # 76 lanes: the 32-column state blocks, a ragged second chunk
    (38, 130, 4),   # 152 lanes: the 64-column state blocks, ragged third chunk
    (75, 1, 1),     # 75 lanes (the 16-column blocks), one step each
    (19, 257, 8),   # 152 lanes over five chunks, the last one step long
])
def test_delta_state_block_widths(B, T, H):
    # the state pass splits the value columns into blocks of 64, 32 or 16 by
    # the lane count; each width, its boundary and a ragged last chunk
    d = {k: (v.cuda() if v is not None else None)
         for k, v in inputs.delta_inputs(B, T, H, 64, seed=1400 + B * T + H, with_S0=True).items()}
    _run(d, T)


@pytest.mark.parametrize("cid,rows", [(13, None), (14, [0, 9, 15]), (15, [0, 15])])
def test_delta_workloads(cid, rows):
    w = inputs.EXTRA_WORKLOADS[cid]
    d = {k: (v.cuda() if v is not None else None) for k, v in w.make(device="cpu").items()}
    _run(d, w.T, rows)


def test_delta_degenerate_and_errors():
    # T = 0: the final state is the initial one; no output rows
    S0 = torch.randn((2, 3, 64, 64), device="cuda")
    e = torch.empty((2, 0, 3, 64), device="cuda")
    o, ST = api.delta_scan_fwd(e, e, e, torch.empty((2, 0, 3), device="cuda"), S0, want_state=True)
    b.mgs_check()
    assert o.shape == e.shape and torch.equal(ST, S0)
    # beta = 0 keeps the state: o_t = S0 q_t
    d = {k: (v.cuda() if v is not None else None) for k, v in inputs.delta_inputs(2, 70, 2, 64, seed=5).items()}
    o = api.delta_scan_fwd(d["q"], d["k"], d["v"], torch.zeros_like(d["beta"]), d["S0"])
    b.mgs_check()
    ref = torch.einsum("bhij,bthj->bthi", d["S0"].double(), d["q"].double())
    assert_close("o (beta = 0)", o, ref.cpu().numpy(), 70)
    # only D = 64
    x = torch.zeros((1, 4, 1, 32), device="cuda")
    with pytest.raises(b.MGSError) as err:
        b.mgs_delta_scan_fwd(x, x.clone(), x.clone(), torch.zeros((1, 4, 1), device="cuda"), None,
                             torch.empty_like(x), None, 1, 4, 1, 32)
    assert err.value.status == b.MGS_ERR_UNSUPPORTED
    # the workspace: required, and disjoint from the outputs
    o = torch.empty_like(d["q"])
    with pytest.raises(b.MGSError) as err:
        b.mgs_delta_scan_fwd(d["q"], d["k"], d["v"], d["beta"], d["S0"], o, None, 2, 70, 2, 64)
    assert err.value.status == b.MGS_ERR_WORKSPACE
    ws, nws = api.workspace(b.MGS_OP_DELTA_SCAN_FWD, 2, 70, 2, 64, "cuda")
    assert nws == 2 * 2 * 2 * 4 * 64 * 64 * 4
    with pytest.raises(b.MGSError) as err:
        b.mgs_delta_scan_fwd(d["q"], d["k"], d["v"], d["beta"], d["S0"], o, None, 2, 70, 2, 64, ws, nws // 2)
    assert err.value.status == b.MGS_ERR_WORKSPACE
    big = torch.empty(nws // 4 + o.numel(), device="cuda")
    with pytest.raises(b.MGSError) as err:
        b.mgs_delta_scan_fwd(d["q"], d["k"], d["v"], d["beta"], d["S0"], big[:o.numel()].view(o.shape), None,
                             2, 70, 2, 64, big, nws)
    assert err.value.status == b.MGS_ERR_INVALID_ARG
