"""The oracle pins catch plausible mistakes (CPU only).

Each case plants one mistake in a COPY of oracle/moe_oracle.c inside a
temporary directory, runs the pin suite against that copy in a subprocess and
expects failures.  The real oracle is never modified."""
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

MUTATIONS = {
    "tie_to_higher_id": ("return a < b; /* equal", "return a > b; /* equal"),
    "silu_sign": ("return z / (1.0 + exp(-z));", "return z / (1.0 + exp(z));"),
    "gate_reads_up": ("g += load_elem(gate, wdt, base + h) * x[h];",
                      "g += load_elem(up, wdt, base + h) * x[h];"),
    "down_transposed": ("int64_t base = (e * H + c) * I;", "int64_t base = (e * I + c) * H;"),
    "unstable_dispatch": ("for (int64_t s = 0; s < n; ++s) { /* ascending s: stable */",
                          "for (int64_t s = n - 1; s >= 0; --s) {"),
    "plus_inf_not_poison": ("if (l[e] == INFINITY) has_pinf = 1;", ";"),
    "renorm_dropped": ("for (int j = 0; j < k; ++j) w_pre[j] = w_pre[j] / tot;", ";"),
    "combine_unweighted": ("w_cast[t * k + j] * expert_out[r * H + c]", "expert_out[r * H + c]"),
    "softmax_without_max_shift": ("    double s = 0.0;\n    for (int64_t e = 0; e < E; ++e) s += exp(l[e] - m);",
                                  "    double s = 0.0;\n    for (int64_t e = 0; e < E; ++e) s += exp(l[e]);"),
    "sigmoid_bias_in_weights": ("sig[e] = 1.0 / (1.0 + exp(-l));",
                                "sig[e] = 1.0 / (1.0 + exp(-l)) + (bias ? bias[e] : 0.0);"),
    "sigmoid_top_two_ignored": ("gscore[g] = group_top_two ? best + second : best;",
                                "gscore[g] = best;"),
    "sigmoid_group_tie_to_higher": ("if (!gsel[g] && (bg < 0 || beats_f(gscore[g], g, gscore[bg], bg))) bg = g;",
                                    "if (!gsel[g] && (bg < 0 || gscore[g] >= gscore[bg])) bg = g;"),
    "silu_grad_wrong": ("return s * (1.0 + z * (1.0 - s));", "return s * (1.0 + z * s);"),
    "dgate_missing_up_factor": ("const double dg = d * uu * silu_grad(gg);", "const double dg = d * silu_grad(gg);"),
    "router_renorm_sign": ("c[m] = renorm ? scale * (dw[t * k + m] / Q - gq / (Q * Q)) : scale * dw[t * k + m];",
                           "c[m] = renorm ? scale * (dw[t * k + m] / Q + gq / (Q * Q)) : scale * dw[t * k + m];"),
    "combine_backward_unweighted": ("dexpert[r * H + h] = w[s] * dy[t * H + h];", "dexpert[r * H + h] = dy[t * H + h];"),
    "dup_weight_grad_without_silu": ("const double cg = d * uu * silu_grad(gg), cu = d * silu(gg);",
                                     "const double cg = d * uu * silu_grad(gg), cu = d * uu;"),
    "ddown_weight_grad_without_up": ("sd[i] += dd * sl[r * I + i] * u[r * I + i];",
                                     "sd[i] += dd * sl[r * I + i];"),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_planted_mistake(tmp_path, name):
    old, new = MUTATIONS[name]
    src = open(os.path.join(ROOT, "oracle", "moe_oracle.c")).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not found exactly once"
    root = tmp_path / "repo"
    shutil.copytree(os.path.join(ROOT, "oracle"), root / "oracle",
                    ignore=shutil.ignore_patterns("_build", "__pycache__"))
    shutil.copytree(os.path.join(ROOT, "tests"), root / "tests",
                    ignore=shutil.ignore_patterns("__pycache__"))
    (root / "oracle" / "moe_oracle.c").write_text(src.replace(old, new))
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-p", "no:cacheprovider",
                        "tests/test_oracle_pins.py", "tests/test_oracle_sigmoid_pins.py",
                        "tests/test_oracle_backward_pins.py"],
                       cwd=root, capture_output=True, text=True,
                       timeout=600)
    tail = r.stdout.strip().splitlines()[-1] if r.stdout.strip() else r.stderr[-500:]
    assert r.returncode != 0 and "failed" in tail, f"{name} went unnoticed: {tail}"
