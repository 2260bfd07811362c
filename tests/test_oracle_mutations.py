"""Plants plausible mistakes in a copy of the oracle's C source (a transposed
operand, a dropped term, a wrong index or sign), builds each copy on the CPU
and checks that the pin suite rejects every one of them."""
import os
import subprocess
import sys

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(os.path.dirname(HERE), "oracle", "mgs_oracle.c")

# (name, text in mgs_oracle.c, replacement, occurrence index)
MUTATIONS = [
    ("mas_fwd_transposed_A", "s += At[i * K + j] * prev[j];", "s += At[j * K + i] * prev[j];", 0),
    ("mas_fwd_dropped_b", "double s = bt[i];", "double s = 0.0;", 0),
    ("mas_bwd_untransposed_A", "s += At[i * K + j] * lam[i];", "s += At[j * K + i] * lam[i];", 0),
    ("mas_bwd_dA_uses_h_t", "dAt[i * K + j] = lam[i] * states[(t - 1) * K + j];",
     "dAt[i * K + j] = lam[i] * states[t * K + j];", 0),
    ("mas_bwd_dropped_carry", "lam[i] = gt[i] + nxt[i];", "lam[i] = gt[i];", 0),
    ("ms_fwd_right_multiply", "s += At[i * K + m] * prev[m * K + j];",
     "s += prev[i * K + m] * At[m * K + j];", 0),
    ("ms_bwd_P_not_transposed", "s += lam[i * K + j] * Pprev[m * K + j];",
     "s += lam[i * K + j] * Pprev[j * K + m];", 0),
    ("psl_fwd_wrong_sign", "log1p(exp(-fabs(x - y)))", "log1p(exp(fabs(x - y)))", 0),
    ("psl_bwd_dlc_uses_h_t", "dlc[idx] = lam * a * hs[t - 1];", "dlc[idx] = lam * a * hs[t];", 0),
    ("psl_bwd_dropped_carry", "lam = gh[idx] + nxt;", "lam = gh[idx];", 0),
    ("linear_fwd_dropped_b", "x = a[idx] * x + bv[idx];", "x = a[idx] * x;", 0),
    ("linear_bwd_da_uses_h_t", "da[idx] = lam * hs[t - 1];", "da[idx] = lam * hs[t];", 0),
    ("givens_rotation_sign", "M[p * K + col] = c * x - s * y;", "M[p * K + col] = c * x + s * y;", 0),
    ("givens_layer_parity", "(l % 2 == 1) ? 0 : 1", "(l % 2 == 1) ? 1 : 0", 0),
    ("givens_layer_order", "for (int64_t l = 1; l <= K; ++l) {", "for (int64_t l = K; l >= 1; --l) {", 0),
    ("givens_deriv_sign", "M[p * K + col] = -s * x - c * y;", "M[p * K + col] = s * x - c * y;", 0),
    ("givens_deriv_keeps_other_rows", "M[r * K + col] = 0.0;", "M[r * K + col] = M[r * K + col];", 0),
    ("gas_fwd_drops_a", "givens_matrix(theta + st * N, a ? a + st * K : NULL, K, -1, M);",
     "givens_matrix(theta + st * N, NULL, K, -1, M);", 0),
    ("gas_bwd_da_uses_A", "givens_matrix(th, NULL, K, -1, M);", "givens_matrix(th, at, K, -1, M);", 0),
    ("gas_bwd_dropped_carry", "lam[i] = gh[st * K + i] + nxt[i];", "lam[i] = gh[st * K + i];", 0),
    ("gms_bwd_P_not_transposed", "s += lam[i * K + j] * Pprev[m * K + j];",
     "s += lam[i * K + j] * Pprev[j * K + m];", 1),
    ("delta_dropped_beta", "S[i * D + j] += bt * (vt[i] - Sk[i]) * kt[j];",
     "S[i * D + j] += (vt[i] - Sk[i]) * kt[j];", 0),
    ("delta_no_erase", "S[i * D + j] += bt * (vt[i] - Sk[i]) * kt[j];",
     "S[i * D + j] += bt * vt[i] * kt[j];", 0),
    ("delta_state_transposed", "s += S[i * D + j] * kt[j];", "s += S[j * D + i] * kt[j];", 0),
    ("delta_state_never_updated", "for (int64_t i = 0; i < D; ++i)\n                for (int64_t j = 0; j < D; ++j)\n"
     "                    S[i * D + j] += bt", "for (int64_t i = 0; i < 0; ++i)\n                for (int64_t j = 0; j < D; ++j)\n"
     "                    S[i * D + j] += bt", 0),
]
PIN_FILES = ["test_oracle_pins.py", "test_oracle_givens_pins.py", "test_oracle_delta_pins.py"]


def _mutate(text, old, new, occ):
    pos = -1
    for _ in range(occ + 1):
        pos = text.index(old, pos + 1)
    return text[:pos] + new + text[pos + len(old):]


@pytest.mark.parametrize("name,old,new,occ", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_pins_reject_planted_mistake(tmp_path, name, old, new, occ):
    src = open(SRC).read()
    mutated = _mutate(src, old, new, occ)
    assert mutated != src
    c = tmp_path / "mut.c"
    c.write_text(mutated)
    so = tmp_path / "libmut.so"
    subprocess.run(["gcc", "-O2", "-fopenmp", "-shared", "-fPIC", "-std=c11", "-o", str(so), str(c), "-lm"],
                   check=True)
    env = dict(os.environ, MGS_ORACLE_LIB=str(so))
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider"]
                       + [os.path.join(HERE, f) for f in PIN_FILES],
                       env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"mutation {name} survived the pins:\n{r.stdout[-2000:]}"
