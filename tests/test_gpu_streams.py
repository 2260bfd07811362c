"""Every entry point honours the stream it is given: the same calls issued on a
side stream (while the default stream is busy with unrelated work) and on the
default stream give the same results, bit for bit (the time-chunked path
included: its three launches add in a fixed order)."""
import pytest
import torch

from scan_linear_recurrences_gb300 import _binding as b
from scan_linear_recurrences_gb300 import api, inputs
from scan_linear_recurrences_gb300.build import build

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    build()
    b.lib()
    yield
    b.mgs_check()


def _cuda(d):
    return {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in d.items()}


def _calls():
    m = _cuda(inputs.mas_inputs(4, 200, 3, 8, seed=31, h0="normal"))
    mc = _cuda(inputs.mas_inputs(2, 700, 3, 8, seed=32, h0="normal"))  # few lanes: time-chunked
    p = _cuda(inputs.psl_inputs(2, 300, 256, seed=33))
    g = _cuda(inputs.givens_affine_inputs(4, 90, 5, 8, seed=34, h0="normal"))
    d = _cuda(inputs.delta_inputs(2, 150, 2, 64, seed=35))

    def run(stream):
        out = {}
        h = api.matrix_affine_scan_fwd(m["A"], m["b"], m["h0"], stream=stream)
        out["mas"] = (h,) + api.matrix_affine_scan_bwd(m["A"], m["h0"], h, m["grad_h"], stream=stream)[:2]
        out["mas_recompute"] = api.matrix_affine_scan_bwd_recompute(m["A"], m["b"], m["h0"], m["grad_h"],
                                                                    stream=stream)[:2]
        hc = api.matrix_affine_scan_fwd(mc["A"], mc["b"], mc["h0"], stream=stream)
        out["mas_chunked"] = (hc,) + api.matrix_affine_scan_bwd(mc["A"], mc["h0"], hc, mc["grad_h"], stream=stream)[:2]
        hp = api.parallel_scan_log_fwd(p["log_coeffs"], p["log_values"], p["log_h0"], stream=stream)
        out["psl"] = (hp,) + api.parallel_scan_log_bwd(p["log_coeffs"], p["log_values"], p["log_h0"], None,
                                                       p["grad_h"], stream=stream)[:2]
        hg = api.givens_affine_scan_fwd(g["theta"], g["a"], g["b"], g["h0"], stream=stream)
        out["givens"] = (hg,) + api.givens_affine_scan_bwd(g["theta"], g["a"], g["h0"], hg, g["grad_h"],
                                                           stream=stream)[:2]
        out["delta"] = api.delta_scan_fwd(d["q"], d["k"], d["v"], d["beta"], d["S0"], want_state=True, stream=stream)
        return out
    return run


def test_side_stream_matches_default_stream():
    run = _calls()
    ref = run(None)
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    busy = torch.empty(64 << 20, device="cuda")
    with torch.cuda.stream(side):
        busy.normal_()                      # unrelated work on the same stream first
        got = run(side.cuda_stream)
    b.mgs_check(side.cuda_stream)
    side.synchronize()
    for name in ref:
        for x, y in zip(ref[name], got[name]):
            assert torch.equal(x, y), name
