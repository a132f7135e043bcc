"""The pins must catch plausible mistakes in the oracle.

Each case plants one mistake in a copy of the oracle's C source (on the CPU, in a temporary
directory), builds it, and runs the pin suite against it: the suite must fail.  The real
oracle is never modified.
"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "gdn_oracle.c")

MUTATIONS = {
    "no_decay": ("for (int j = 0; j < dk; ++j) s[j] *= decay;",
                 "for (int j = 0; j < dk; ++j) s[j] *= 1.0;"),
    "no_beta": ("double delta = beta * (v[i] - kv);", "double delta = (v[i] - kv);"),
    "read_before_decay": ("double decay = exp(g);", "double decay = 1.0;"),
    "output_before_write": ("for (int j = 0; j < dk; ++j) s[j] += delta * k[j];          /* 4. write */\n    double acc = 0.0;\n    for (int j = 0; j < dk; ++j) acc += s[j] * q[j];            /* 5. output */",
                            "double acc = 0.0;\n    for (int j = 0; j < dk; ++j) acc += s[j] * q[j];\n    for (int j = 0; j < dk; ++j) s[j] += delta * k[j];"),
    "softplus_sign": ("return fmax(x, 0.0) + log1p(exp(-fabs(x)));",
                      "return fmax(x, 0.0) + log1p(exp(fabs(x))) - fabs(x);"),
    "gate_sign": ("return -exp(A_log) * gdn_oracle_softplus(a + dt_bias);",
                  "return -exp(A_log) * gdn_oracle_softplus(a - dt_bias);"),
    "chunk_mask_sign": ("val = bb[r] * exp(G[r] - G[s]) * kk;",
                        "val = bb[r] * exp(G[s] - G[r]) * kk;"),
    "chunk_u_sign": ("U[(size_t)r * dv + i] = Up[(size_t)r * dv + i] - s_;",
                     "U[(size_t)r * dv + i] = Up[(size_t)r * dv + i] + s_;"),
    "chunk_drop_inter": ("o[(size_t)(t0 + r) * dv + i] = exp(G[r]) * inter + intra;",
                         "o[(size_t)(t0 + r) * dv + i] = intra;"),
    "solve_skip_row": ("for (int s = 0; s < r; ++s) {\n      double a = A[(size_t)r * n + s];",
                       "for (int s = 0; s + 1 < r; ++s) {\n      double a = A[(size_t)r * n + s];"),
    "conv_taps_reversed": ("y += w[(size_t)c * W + j] * conv_input",
                           "y += w[(size_t)c * W + (W - 1 - j)] * conv_input"),
    "gqa_map_modulo": ("int W = c->conv_width, r = Hv / Hk, kh = h / r;",
                       "int W = c->conv_width, r = Hv / Hk, kh = h % Hk;"),
    "l2norm_no_sqrt": ("double inv = scale / sqrt(ss + eps);", "double inv = scale / (ss + eps);"),
    "conv_state_off_by_one": ("int idx = (W - 1) + tau;", "int idx = (W - 2) + tau;"),
    "rmsnorm_sum_not_mean": ("ms /= (double)n;", "ms /= 1.0;"),
    "rmsnorm_no_sqrt": ("double inv = 1.0 / sqrt(ms + eps);", "double inv = 1.0 / (ms + eps);"),
    "rmsnorm_gate_sign": ("double gate = zrow[i] * gdn_oracle_sigmoid(zrow[i]);",
                          "double gate = zrow[i] * gdn_oracle_sigmoid(-zrow[i]);"),
    "rmsnorm_no_weight": ("y[(size_t)r * n + i] = w[i] * (orow[i] * inv) * gate;",
                          "y[(size_t)r * n + i] = (orow[i] * inv) * gate;"),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_planted_mistake(name, tmp_path):
    old, new = MUTATIONS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not found exactly once"
    mut = tmp_path / "gdn_oracle_mut.c"
    mut.write_text(src.replace(old, new))
    lib = tmp_path / "liboracle_mut.so"
    subprocess.run(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-o", str(lib), str(mut),
                    "-lm", "-lpthread"], check=True)
    env = dict(os.environ, GDN_ORACLE_LIB=str(lib))
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                       env=env, cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode != 0, f"planted mistake '{name}' passed every pin:\n{r.stdout[-2000:]}"
