"""The no-allocation matrix_scan forward (mgs_matrix_scan_fwd_noalloc).

It serves callers that own only their input and output buffers and cannot call
cudaMalloc (device memory owned by another runtime's pool allocator, or a
latency-bound loop that cannot take cudaMalloc's device-wide synchronisation):
its scratch is a fixed-size device array inside the library.  This file is
named so that pytest collects it last.
"""
import pytest
import torch

import oracle
from scan_linear_recurrences_gb300 import _binding as b
from scan_linear_recurrences_gb300 import inputs
from scan_linear_recurrences_gb300.build import build

from ._parity import assert_close

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("B,T,H,k,uses_scratch", [
    (16, 1024, 8, 8, True),   # time-chunked: carries go through the built-in scratch
    (1, 333, 2, 8, True),     # chunked, ragged last chunk
    (2, 1000, 3, 4, True),
    (4, 48, 8, 8, False),     # short sequence: single pass, no scratch needed
])
def test_noalloc_matches_the_oracle_on_two_calls(B, T, H, k, uses_scratch):
    build()
    b.lib()
    d = inputs.ms_inputs(B, T, H, k, seed=900 + T)
    n = b.mgs_workspace_size(b.MGS_OP_MATRIX_SCAN_FWD, B, T, H, k)
    assert n <= b.NOALLOC_SCRATCH_BYTES
    # the chunked shapes must really exercise the library's own scratch array
    assert (n > 0) == uses_scratch
    ref = oracle.ms_fwd(d["A"])
    A = d["A"].cuda()
    # two calls in a row through the C ABI; the second reuses the scratch the first left behind
    P1 = torch.full_like(A, float("nan"))
    P2 = torch.full_like(A, float("nan"))
    b.mgs_matrix_scan_fwd_noalloc(A, P1, B, T, H, k)
    b.mgs_matrix_scan_fwd_noalloc(A, P2, B, T, H, k)
    b.mgs_check()
    assert_close("first call", P1, ref, T)
    assert_close("second call", P2, ref, T)


def test_noalloc_rejects_shapes_beyond_the_scratch():
    build()
    # k = 16, one lane group, very long sequence: more carry scratch than the array holds
    B, T, H, k = 1, 131072, 2, 16
    assert b.mgs_workspace_size(b.MGS_OP_MATRIX_SCAN_FWD, B, T, H, k) > b.NOALLOC_SCRATCH_BYTES
    fake = 1 << 40  # never dereferenced: the size check comes first
    with pytest.raises(b.MGSError) as ei:
        b.mgs_matrix_scan_fwd_noalloc(fake, fake + (1 << 36), B, T, H, k, stream=0)
    assert ei.value.status == b.MGS_ERR_WORKSPACE
