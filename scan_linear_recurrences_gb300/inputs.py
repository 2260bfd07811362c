"""Seeded synthetic inputs for the scan primitives.

This module holds no scan arithmetic: it only draws random numbers and shapes
them into the input tensors that both the CUDA library and the float64 oracle
receive.  Every tensor is produced in float64 on the chosen device and cast to
float32 at the end, so the oracle (which upcasts float32 exactly) and the GPU
see bit-identical inputs.

Workloads follow the shapes the mingru-scans pages benchmark ("Run the
benchmarks", Step 2: the lab shape B=128, T=64 and the long-sequence shape
T=1024; the home page's table gives B=16 for long-T and d=64, k=8 for the
GivensMinGRU memory row) plus a scaled throughput shape and the minGRU
log-space gate distribution.

Recipes (each draws from one ``torch.Generator`` seeded with ``seed``, in the
order written; time is generated in blocks of ``TIME_BLOCK`` steps so device
memory stays bounded; within a block the draws are in the order listed):

* matrix_affine_scan: per (b, t, head): G ~ N(0,1)^{k x k}; Q = the
  orthogonal factor of G with positive diagonal R (Haar on O(k), Mezzadri
  2007), a = sigmoid(N(0,1))^k, A = Q diag(a); z = sigmoid(N(0,1))^k,
  n = N(0,1)^k, b = z * n; grad_h = N(0,1)^k.  h0 is drawn before the time
  blocks when requested (N(0,1)), else absent (zero initial state).
* matrix_scan: A_t = L_k ... L_1, a brick-wall mesh of k layers of 2x2 Givens
  rotations on adjacent coordinates (odd layers (0,1),(2,3),...; even layers
  (1,2),(3,4),...; no wrap), each angle ~ U(-pi, pi), k(k-1)/2 angles per
  matrix; rotation on (i, i+1) maps (x_i, x_{i+1}) to
  (c x_i - s x_{i+1}, s x_i + c x_{i+1}).  grad_P = N(0,1)^{k x k}.
* Givens affine scan (GivensMinGRU transition from its angles): h0 as for
  matrix_affine_scan; per block theta ~ U(-pi, pi)^{k(k-1)/2}, a =
  sigmoid(N(0,1))^k (drawn even when the op is run without a), z =
  sigmoid(N(0,1))^k, n = N(0,1)^k, b = z * n, grad_h = N(0,1)^k.
* Givens matrix scan: per block theta ~ U(-pi, pi)^{k(k-1)/2} (the angles
  of the matrix_scan recipe above), grad_P = N(0,1)^{k x k}.
* delta rule (DeltaNet, behind DeltaMinGRU): S0 = N(0,1)^{DxD}/sqrt(D) drawn
  first when requested; per block q ~ N(0,1)^D normalised, k likewise, v =
  N(0,1)^D, beta = sigmoid(N(0,1)) per (b, t, head).
* parallel_scan_log (minGRU gates): log_h0 = log g(N(0,1)) drawn first; then
  per block u ~ N(0,1), x ~ N(0,1), grad_h ~ N(0,1);
  log_coeffs = log(1 - sigmoid(u)) = -softplus(u),
  log_values = log(sigmoid(u)) + log g(x) = -softplus(-u) + log g(x),
  with g(x) = x + 0.5 for x >= 0 and sigmoid(x) otherwise.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import torch

TIME_BLOCK = 256
BASE_SEED = 20261202


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=torch.device(device))
    g.manual_seed(int(seed))
    return g


def haar_orthogonal(G: torch.Tensor) -> torch.Tensor:
    """Orthogonal factor Q of G = QR with R's diagonal positive, batched over the
    leading dims of G [..., k, k] (float64).  Computed column by column with
    classical Gram-Schmidt applied twice (re-orthogonalisation), which yields the
    same Q as Householder QR followed by the sign fix Q <- Q diag(sign diag R)."""
    k = G.shape[-1]
    cols = []
    for j in range(k):
        v = G[..., :, j]
        for _ in range(2):
            for q in cols:
                v = v - (q * v).sum(-1, keepdim=True) * q
        v = v / torch.linalg.vector_norm(v, dim=-1, keepdim=True)
        cols.append(v)
    return torch.stack(cols, dim=-1)


def givens_mesh(theta: torch.Tensor, k: int) -> torch.Tensor:
    """Brick-wall product of Givens rotations.  theta [..., k(k-1)/2] (float64)
    -> A [..., k, k] = L_k ... L_1, layer 1 applied first."""
    lead = theta.shape[:-1]
    M = torch.eye(k, dtype=theta.dtype, device=theta.device).expand(*lead, k, k).clone()
    idx = 0
    for layer in range(1, k + 1):
        first = 0 if layer % 2 == 1 else 1
        for i in range(first, k - 1, 2):
            c = torch.cos(theta[..., idx]).unsqueeze(-1)
            s = torch.sin(theta[..., idx]).unsqueeze(-1)
            ri = M[..., i, :].clone()
            rj = M[..., i + 1, :].clone()
            M[..., i, :] = c * ri - s * rj
            M[..., i + 1, :] = s * ri + c * rj
            idx += 1
    assert idx == k * (k - 1) // 2
    return M


def _g_of_x(x: torch.Tensor) -> torch.Tensor:
    return torch.where(x >= 0, x + 0.5, torch.sigmoid(x))


def _log_g_of_x(x: torch.Tensor) -> torch.Tensor:
    # log(x + 0.5) on x >= 0, log sigmoid(x) = -softplus(-x) on x < 0
    return torch.where(x >= 0, torch.log(torch.clamp(x, min=0) + 0.5),
                       -torch.nn.functional.softplus(-x))


def mas_inputs(B, T, H, k, seed, device="cpu", h0="none"):
    """matrix_affine_scan inputs: dict(A [B,T,H,k,k], b [B,T,H,k], h0 [B,H,k] or
    None, grad_h [B,T,H,k]), float32 on ``device``.  ``h0``: "none" (zero
    initial state, passed as absent), "zeros" (explicit zeros) or "normal"."""
    dev = torch.device(device)
    g = _gen(seed, dev)
    f64 = dict(dtype=torch.float64, device=dev)
    A = torch.empty((B, T, H, k, k), dtype=torch.float32, device=dev)
    b = torch.empty((B, T, H, k), dtype=torch.float32, device=dev)
    gh = torch.empty((B, T, H, k), dtype=torch.float32, device=dev)
    if h0 == "normal":
        h0_t = torch.randn((B, H, k), generator=g, **f64).float()
    elif h0 == "zeros":
        h0_t = torch.zeros((B, H, k), dtype=torch.float32, device=dev)
    elif h0 == "none":
        h0_t = None
    else:
        raise ValueError(h0)
    for t0 in range(0, T, TIME_BLOCK):
        tb = min(TIME_BLOCK, T - t0)
        G = torch.randn((B, tb, H, k, k), generator=g, **f64)
        Q = haar_orthogonal(G)
        a = torch.sigmoid(torch.randn((B, tb, H, k), generator=g, **f64))
        A[:, t0:t0 + tb] = (Q * a.unsqueeze(-2)).float()  # Q diag(a): column j scaled by a_j
        z = torch.sigmoid(torch.randn((B, tb, H, k), generator=g, **f64))
        n = torch.randn((B, tb, H, k), generator=g, **f64)
        b[:, t0:t0 + tb] = (z * n).float()
        gh[:, t0:t0 + tb] = torch.randn((B, tb, H, k), generator=g, **f64).float()
    return dict(A=A, b=b, h0=h0_t, grad_h=gh)


def ms_inputs(B, T, H, k, seed, device="cpu"):
    """matrix_scan inputs: dict(A [B,T,H,k,k] Givens brick-wall meshes,
    grad_P [B,T,H,k,k]), float32 on ``device``."""
    dev = torch.device(device)
    g = _gen(seed, dev)
    f64 = dict(dtype=torch.float64, device=dev)
    nang = k * (k - 1) // 2
    A = torch.empty((B, T, H, k, k), dtype=torch.float32, device=dev)
    gP = torch.empty((B, T, H, k, k), dtype=torch.float32, device=dev)
    for t0 in range(0, T, TIME_BLOCK):
        tb = min(TIME_BLOCK, T - t0)
        theta = (torch.rand((B, tb, H, nang), generator=g, **f64) * 2.0 - 1.0) * math.pi
        A[:, t0:t0 + tb] = givens_mesh(theta, k).float()
        gP[:, t0:t0 + tb] = torch.randn((B, tb, H, k, k), generator=g, **f64).float()
    return dict(A=A, grad_P=gP)


def givens_affine_inputs(B, T, H, k, seed, device="cpu", h0="none", with_a=True):
    """Givens affine scan inputs: dict(theta [B,T,H,k(k-1)/2], a [B,T,H,k] or
    None, b [B,T,H,k], h0 [B,H,k] or None, grad_h [B,T,H,k]), float32."""
    dev = torch.device(device)
    g = _gen(seed, dev)
    f64 = dict(dtype=torch.float64, device=dev)
    nang = k * (k - 1) // 2
    th = torch.empty((B, T, H, nang), dtype=torch.float32, device=dev)
    a = torch.empty((B, T, H, k), dtype=torch.float32, device=dev)
    b = torch.empty((B, T, H, k), dtype=torch.float32, device=dev)
    gh = torch.empty((B, T, H, k), dtype=torch.float32, device=dev)
    if h0 == "normal":
        h0_t = torch.randn((B, H, k), generator=g, **f64).float()
    elif h0 == "none":
        h0_t = None
    else:
        raise ValueError(h0)
    for t0 in range(0, T, TIME_BLOCK):
        tb = min(TIME_BLOCK, T - t0)
        th[:, t0:t0 + tb] = ((torch.rand((B, tb, H, nang), generator=g, **f64) * 2.0 - 1.0) * math.pi).float()
        a[:, t0:t0 + tb] = torch.sigmoid(torch.randn((B, tb, H, k), generator=g, **f64)).float()
        z = torch.sigmoid(torch.randn((B, tb, H, k), generator=g, **f64))
        n = torch.randn((B, tb, H, k), generator=g, **f64)
        b[:, t0:t0 + tb] = (z * n).float()
        gh[:, t0:t0 + tb] = torch.randn((B, tb, H, k), generator=g, **f64).float()
    return dict(theta=th, a=a if with_a else None, b=b, h0=h0_t, grad_h=gh)


def givens_matrix_inputs(B, T, H, k, seed, device="cpu"):
    """Givens matrix scan inputs: dict(theta [B,T,H,k(k-1)/2], grad_P [B,T,H,k,k])."""
    dev = torch.device(device)
    g = _gen(seed, dev)
    f64 = dict(dtype=torch.float64, device=dev)
    nang = k * (k - 1) // 2
    th = torch.empty((B, T, H, nang), dtype=torch.float32, device=dev)
    gP = torch.empty((B, T, H, k, k), dtype=torch.float32, device=dev)
    for t0 in range(0, T, TIME_BLOCK):
        tb = min(TIME_BLOCK, T - t0)
        th[:, t0:t0 + tb] = ((torch.rand((B, tb, H, nang), generator=g, **f64) * 2.0 - 1.0) * math.pi).float()
        gP[:, t0:t0 + tb] = torch.randn((B, tb, H, k, k), generator=g, **f64).float()
    return dict(theta=th, grad_P=gP)


def delta_inputs(B, T, H, D, seed, device="cpu", with_S0=True):
    """Delta-rule inputs (DeltaNet conventions): q, k = unit vectors (N(0,1)^D
    normalised), v = N(0,1)^D, beta = sigmoid(N(0,1)); S0 = N(0,1)^{DxD}/sqrt(D)
    drawn first when requested.  dict(q, k, v [B,T,H,D], beta [B,T,H], S0)."""
    dev = torch.device(device)
    g = _gen(seed, dev)
    f64 = dict(dtype=torch.float64, device=dev)
    S0 = (torch.randn((B, H, D, D), generator=g, **f64) / math.sqrt(D)).float() if with_S0 else None
    q = torch.empty((B, T, H, D), dtype=torch.float32, device=dev)
    k = torch.empty_like(q)
    v = torch.empty_like(q)
    beta = torch.empty((B, T, H), dtype=torch.float32, device=dev)
    for t0 in range(0, T, TIME_BLOCK):
        tb = min(TIME_BLOCK, T - t0)
        qq = torch.randn((B, tb, H, D), generator=g, **f64)
        kk = torch.randn((B, tb, H, D), generator=g, **f64)
        q[:, t0:t0 + tb] = (qq / qq.norm(dim=-1, keepdim=True)).float()
        k[:, t0:t0 + tb] = (kk / kk.norm(dim=-1, keepdim=True)).float()
        v[:, t0:t0 + tb] = torch.randn((B, tb, H, D), generator=g, **f64).float()
        beta[:, t0:t0 + tb] = torch.sigmoid(torch.randn((B, tb, H), generator=g, **f64)).float()
    return dict(q=q, k=k, v=v, beta=beta, S0=S0)


def psl_inputs(B, T, D, seed, device="cpu", with_h0=True):
    """parallel_scan_log inputs with the minGRU gate distribution:
    dict(log_coeffs, log_values [B,T,D], log_h0 [B,D] or None, grad_h [B,T,D])."""
    dev = torch.device(device)
    g = _gen(seed, dev)
    f64 = dict(dtype=torch.float64, device=dev)
    l0 = _log_g_of_x(torch.randn((B, D), generator=g, **f64)).float() if with_h0 else None
    lc = torch.empty((B, T, D), dtype=torch.float32, device=dev)
    lv = torch.empty((B, T, D), dtype=torch.float32, device=dev)
    gh = torch.empty((B, T, D), dtype=torch.float32, device=dev)
    for t0 in range(0, T, TIME_BLOCK):
        tb = min(TIME_BLOCK, T - t0)
        u = torch.randn((B, tb, D), generator=g, **f64)
        x = torch.randn((B, tb, D), generator=g, **f64)
        lc[:, t0:t0 + tb] = (-torch.nn.functional.softplus(u)).float()
        lv[:, t0:t0 + tb] = (-torch.nn.functional.softplus(-u) + _log_g_of_x(x)).float()
        gh[:, t0:t0 + tb] = torch.randn((B, tb, D), generator=g, **f64).float()
    return dict(log_coeffs=lc, log_values=lv, log_h0=l0, grad_h=gh)


def linear_inputs(B, T, D, seed, device="cpu", with_h0=True):
    """linear_scan inputs with signed gates: a = tanh(N(0,1)) in (-1, 1),
    b = sigmoid(N(0,1)) * N(0,1), h0 ~ N(0,1) (drawn first) or absent,
    grad_h ~ N(0,1); dict(a, b [B,T,D], h0 [B,D] or None, grad_h)."""
    dev = torch.device(device)
    g = _gen(seed, dev)
    f64 = dict(dtype=torch.float64, device=dev)
    h0 = torch.randn((B, D), generator=g, **f64).float() if with_h0 else None
    a = torch.empty((B, T, D), dtype=torch.float32, device=dev)
    b = torch.empty((B, T, D), dtype=torch.float32, device=dev)
    gh = torch.empty((B, T, D), dtype=torch.float32, device=dev)
    for t0 in range(0, T, TIME_BLOCK):
        tb = min(TIME_BLOCK, T - t0)
        a[:, t0:t0 + tb] = torch.tanh(torch.randn((B, tb, D), generator=g, **f64)).float()
        z = torch.sigmoid(torch.randn((B, tb, D), generator=g, **f64))
        b[:, t0:t0 + tb] = (z * torch.randn((B, tb, D), generator=g, **f64)).float()
        gh[:, t0:t0 + tb] = torch.randn((B, tb, D), generator=g, **f64).float()
    return dict(a=a, b=b, h0=h0, grad_h=gh)


@dataclass(frozen=True)
class Workload:
    """One benchmarked shape."""
    cid: int
    op: str          # "mas" | "ms" | "psl" | "lin" | "gas" | "gms" | "delta"
    name: str
    B: int
    T: int
    H: int           # heads (mas/ms) or channels D (psl)
    k: int           # block size (1 for psl)
    h0: str          # "none" | "normal" for mas; "log" for psl

    @property
    def seed(self) -> int:
        return BASE_SEED + self.cid

    def make(self, device="cpu"):
        if self.op == "mas":
            return mas_inputs(self.B, self.T, self.H, self.k, self.seed, device, h0=self.h0)
        if self.op == "ms":
            return ms_inputs(self.B, self.T, self.H, self.k, self.seed, device)
        if self.op == "lin":
            return linear_inputs(self.B, self.T, self.H, self.seed, device, with_h0=True)
        if self.op == "gas":
            return givens_affine_inputs(self.B, self.T, self.H, self.k, self.seed, device, h0=self.h0)
        if self.op == "gms":
            return givens_matrix_inputs(self.B, self.T, self.H, self.k, self.seed, device)
        if self.op == "delta":
            return delta_inputs(self.B, self.T, self.H, self.k, self.seed, device, with_S0=True)
        return psl_inputs(self.B, self.T, self.H, self.seed, device, with_h0=True)


WORKLOADS = {
    0: Workload(0, "mas", "matrix_affine_scan small B=2 T=64 H=2 k=8", 2, 64, 2, 8, "none"),
    1: Workload(1, "mas", "matrix_affine_scan lab B=128 T=64 H=8 k=8", 128, 64, 8, 8, "none"),
    2: Workload(2, "ms", "matrix_scan long-T Givens B=16 T=1024 H=8 k=8", 16, 1024, 8, 8, "none"),
    3: Workload(3, "psl", "parallel_scan_log minGRU B=64 T=4096 D=1024", 64, 4096, 1024, 1, "log"),
    4: Workload(4, "mas", "matrix_affine_scan scaled B=32 T=8192 H=64 k=8", 32, 8192, 64, 8, "normal"),
}

# The pages' other benchmark shapes (lab B=128 T=64, long-T B=16 T=1024) for the
# ops the table above covers at one shape only; reported beside the step.
EXTRA_WORKLOADS = {
    5: Workload(5, "mas", "matrix_affine_scan long-T B=16 T=1024 H=8 k=8", 16, 1024, 8, 8, "normal"),
    6: Workload(6, "ms", "matrix_scan lab Givens B=128 T=64 H=8 k=8", 128, 64, 8, 8, "none"),
    7: Workload(7, "lin", "linear_scan lab B=128 T=64 D=64", 128, 64, 64, 1, "normal"),
    8: Workload(8, "lin", "linear_scan long-T B=16 T=1024 D=64", 16, 1024, 64, 1, "normal"),
    # GivensMinGRU's angle-fused scans at the pages' memory-benchmark shape
    # (B=128, T=64, d=64 = 8 heads of k=8) and the long-sequence shape
    9: Workload(9, "gas", "givens_affine_scan lab B=128 T=64 H=8 k=8", 128, 64, 8, 8, "normal"),
    10: Workload(10, "gas", "givens_affine_scan long-T B=16 T=1024 H=8 k=8", 16, 1024, 8, 8, "normal"),
    11: Workload(11, "gms", "givens_matrix_scan lab B=128 T=64 H=8 k=8", 128, 64, 8, 8, "none"),
    12: Workload(12, "gms", "givens_matrix_scan long-T B=16 T=1024 H=8 k=8", 16, 1024, 8, 8, "none"),
    # DeltaMinGRU's delta rule (forward only), head dimension 64 (k holds D):
    # the pages' lab and long-T shapes with one head of d=64, and a throughput
    # shape with enough (batch, head) lanes to fill the GPU
    13: Workload(13, "delta", "delta_scan lab B=128 T=64 H=1 D=64", 128, 64, 1, 64, "normal"),
    14: Workload(14, "delta", "delta_scan long-T B=16 T=1024 H=1 D=64", 16, 1024, 1, 64, "normal"),
    15: Workload(15, "delta", "delta_scan scaled B=16 T=4096 H=16 D=64", 16, 4096, 16, 64, "normal"),
    # parallel_scan_log at the pages' lab and long-T shapes (64 channels)
    16: Workload(16, "psl", "parallel_scan_log lab B=128 T=64 D=64", 128, 64, 64, 1, "log"),
    17: Workload(17, "psl", "parallel_scan_log long-T B=16 T=1024 D=64", 16, 1024, 64, 1, "log"),
    # and at config 3's sequence length with the long-T shape's few lanes
    18: Workload(18, "psl", "parallel_scan_log few-lane B=16 T=4096 D=64", 16, 4096, 64, 1, "log"),
}
