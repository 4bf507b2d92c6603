"""Planted mistakes (CPU only): each plausible error in the C oracle -- a
dropped term, a wrong sign, index or operand, a transposed state -- is planted
into a private copy of gdn_oracle.c, compiled, and run against the pins in
tests/oracle_pins.py.  Every mutant must fail at least one pin; that is the
evidence that the pins constrain every step of the oracle."""
import os
import subprocess
import tempfile

import pytest

import oracle
from tests import oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "gdn_oracle.c")

MUTANTS = {
    "delta_sign": ("const double dj = (v[j] - sj) * beta;", "const double dj = (v[j] + sj) * beta;"),
    "delta_drop_beta": ("const double dj = (v[j] - sj) * beta;", "const double dj = (v[j] - sj);"),
    "update_uses_q": ("St[j * D + i] += dj * k[i];", "St[j * D + i] += dj * q[i];"),
    "drop_scale": ("o[j] = oj * inv_sqrt_d;", "o[j] = oj;"),
    "interleave_heads": ("const int kh = h % Hk;", "const int kh = h / (Hv / Hk);"),
    "taps_reversed": ("u += (double)conv_w[c * KW + j] *", "u += (double)conv_w[c * KW + (KW - 1 - j)] *"),
    "drop_decay": ("for (int i = 0; i < D; ++i) St[j * D + i] *= eg;", "for (int i = 0; i < D; ++i) St[j * D + i] *= 1.0;"),
    "rms_no_mean": ("ms /= (double)D;", "ms /= 1.0;"),
    "rms_eps_outside": ("const double r = 1.0 / sqrt(ms + eps);", "const double r = 1.0 / (sqrt(ms) + eps);"),
    "l2_hf_form": ("nq = sqrt(nq); nk = sqrt(nk);", "nq = sqrt(nq + eps); nk = sqrt(nk + eps);"),
    "drop_dt_bias": ("softplus((double)a_raw[t * Hv + h] + (double)dt_bias[h])", "softplus((double)a_raw[t * Hv + h])"),
    "sk_transposed": ("sj += St[j * D + i] * k[i];", "sj += St[i * D + j] * k[i];"),
    "sq_transposed": ("oj += St[j * D + i] * q[i];", "oj += St[i * D + j] * q[i];"),
    "conv_state_stale": ("const int64_t p = len - 3 + r;", "const int64_t p = len - 4 + r;"),
    "drop_silu_stream": ("    return silu(u);\n}", "    return u;\n}"),
    "gate_no_silu": ("* (double)norm_w[j] * silu((double)z[oi]);", "* (double)norm_w[j] * (double)z[oi];"),
    "gate_sigmoid_z": ("* (double)norm_w[j] * silu((double)z[oi]);", "* (double)norm_w[j] * sigmoid((double)z[oi]);"),
    "drop_norm_w": ("* (double)norm_w[j] * silu((double)z[oi]);", "* silu((double)z[oi]);"),
    "output_reads_k": ("oj += St[j * D + i] * q[i];", "oj += St[j * D + i] * k[i];"),
    "beta_softplus": ("const double beta = sigmoid((double)b_raw[t * Hv + h]);", "const double beta = softplus((double)b_raw[t * Hv + h]);"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor not found exactly once: {old!r}"
    mpath = tmp_path / "mut.c"
    mpath.write_text(src.replace(old, new))
    so = tmp_path / "libmut.so"
    subprocess.run(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-fopenmp", str(mpath),
                    "-o", str(so), "-lm"], check=True)
    lib = oracle.load_library(str(so))
    fwd = lambda **kw: oracle.forward(lib=lib, **kw)
    failed = []
    for check in pins.ALL_CHECKS:
        try:
            check(fwd)
        except AssertionError:
            failed.append(check.__name__)
    assert failed, f"mutant {name} passed every pin"
