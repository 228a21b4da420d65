"""The pins have teeth: plant a plausible mistake in a copy of the oracle's C
source, build it, and check that the pin suite fails on it.

Every mutant lives only in a temporary directory on the CPU; the oracle's
source file is never modified.
"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "attn_oracle.c")

# (name, original text, planted mistake)
MUTANTS = [
    ("dropped_scale", "s[j] = scale * dot + (bias_row", "s[j] = dot + (bias_row"),
    ("bias_wrong_row", "bias + (bias_per_request ? r : flat) * N", "bias + (bias_per_request ? r : flat) * N + 1"),
    ("bias_scaled", "s[j] = scale * dot + (bias_row ? bias_row[j] : 0.0);",
     "s[j] = scale * (dot + (bias_row ? bias_row[j] : 0.0));"),
    ("causal_excludes_diagonal", "*j1 = causal ? i + 1 : N;", "*j1 = causal ? i : N;"),
    ("causal_one_extra_key", "*j1 = causal ? i + 1 : N;", "*j1 = causal ? (i + 2 < N ? i + 2 : N) : N;"),
    ("window_one_extra_key", "i - window + 1 > 0) ? i - window + 1 : 0;",
     "i - window > 0) ? i - window : 0;"),
    ("window_ignored", "*j0 = (causal && window > 0", "*j0 = (causal && window > 1000000"),
    ("dkv_window_one_extra_query", "(causal && window > 0 && j + window < N) ? j + window : N;",
     "(causal && window > 0 && j + window + 1 < N) ? j + window + 1 : N;"),
    ("gqa_modulo_mapping", "const int64_t g = h / group;\n            const double *q_row",
     "const int64_t g = h % Hkv;\n            const double *q_row"),
    ("no_max_subtraction", "const double p = exp(s[t] - m) / l;", "const double p = exp(s[t]) / l;"),
    ("lse_base2", "if (lse) lse[r] = m + log(l);", "if (lse) lse[r] = m + log2(l);"),
    ("lse_missing_max", "if (lse) lse[r] = m + log(l);", "if (lse) lse[r] = log(l);"),
    ("ds_sign_dq", "const double ds = p * (dp - delta[flat]) +", "const double ds = p * (delta[flat] - dp) +"),
    ("ds_sign_dk", "const double ds = p * (dp - delta[qflat]) +", "const double ds = p * (delta[qflat] - dp) +"),
    ("dq_missing_delta", "const double ds = p * (dp - delta[flat]) +", "const double ds = p * dp +"),
    ("dq_drops_grad_in", "(grad_in ? grad_in[flat * N + j] : 0.0);", "0.0;"),
    ("dkv_drops_bias", "const double b_ij = bias ? bias[qflat * N + j] : 0.0;", "const double b_ij = 0.0;"),
    ("dkv_grad_in_transposed", "(grad_in ? grad_in[qflat * N + j] : 0.0);",
     "(grad_in ? grad_in[(qflat - i + j) * N + i] : 0.0);"),
    ("dq_missing_scale", "dq_row[d] += scale * ds * k_head[j * D + d];", "dq_row[d] += ds * k_head[j * D + d];"),
    ("dk_transposed_operand", "dk_row[d] += scale * ds * q_row[d];", "dk_row[d] += scale * ds * do_row[d];"),
    ("dv_uses_ds", "dv_row[d] += p * do_row[d];", "dv_row[d] += ds * do_row[d];"),
    ("dkv_causal_off_by_one", "const int64_t i0 = causal ? j : 0;", "const int64_t i0 = causal ? j + 1 : 0;"),
    ("delta_wrong_operand", "acc += dO[flat * D + d] * o[r * D + d];", "acc += dO[flat * D + d] * dO[flat * D + d];"),
]


@pytest.mark.parametrize("name,orig,bad", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_planted_mistake(tmp_path, name, orig, bad):
    src = open(SRC).read()
    assert src.count(orig) == 1, f"mutation site for {name} not unique"
    mutant_c = tmp_path / "mutant.c"
    mutant_c.write_text(src.replace(orig, bad))
    lib = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O1", "-std=c11", "-fopenmp", "-fPIC", "-shared", str(mutant_c),
                    "-o", str(lib), "-lm"], check=True)
    env = dict(os.environ, TATTN_ORACLE_LIB=str(lib), OMP_NUM_THREADS="2")
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"pins did not catch mutant {name}:\n{r.stdout[-2000:]}"
    assert "failed" in r.stdout, r.stdout[-2000:]
