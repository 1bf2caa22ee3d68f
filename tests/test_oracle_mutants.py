"""Pin strength: plant one plausible mistake at a time in a copy of the oracle's
source, build it, and check that at least one pin fails.  Runs on the CPU;
each mutant runs in its own process so a bad mutant cannot take the test
session down."""
import os
import subprocess
import sys

import pytest

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)

# (name, text in moe_oracle.c, replacement)
MUTANTS = [
    ("gate_sign", "z += exp((double)l[chosen[j]] - l0);", "z += exp(l0 - (double)l[chosen[j]]);"),
    ("gate_numerator", "g[j] = exp((double)l[chosen[j]] - l0) / z;", "g[j] = 1.0 / z;"),
    ("tie_to_higher_index", "if (best < 0 || l[e] > l[best])", "if (best < 0 || l[e] >= l[best])"),
    ("silu_sign", "h[c] = u / (1.0 + exp(-u)) * v;", "h[c] = u / (1.0 + exp(u)) * v;"),
    ("gate_up_swapped", "h[c] = u / (1.0 + exp(-u)) * v;", "h[c] = v / (1.0 + exp(-v)) * u;"),
    ("no_silu", "h[c] = u / (1.0 + exp(-u)) * v;", "h[c] = u * v;"),
    ("w2_transposed", "y += elem(W2[e], wo + (size_t)c, dt) * h[c];",
     "y += elem(W2[e], (size_t)c * d + (size_t)n, dt) * h[c];"),
    ("gate_dropped", "acc[n] += g[j] * y;", "acc[n] += y;"),
    ("accumulate_overwrites", "acc[n] += g[j] * y;", "acc[n] = g[j] * y;"),
    ("bias_ignored", "s += (double)bias[e];", "s += 0.0;"),
    ("router_weight_index", "elem(Wg, (size_t)e * d + i, dt)", "elem(Wg, (size_t)i, dt)"),
    ("perm_token_only", "perm[r] = t * k + j;", "perm[r] = t;"),
    ("route_token_major", "for (int e = 0; e < E; ++e)\n        for (int t = 0; t < T; ++t)\n            for (int j = 0; j < k; ++j)\n                if (idx_out[(size_t)t * k + j] == e) {",
     "for (int t = 0; t < T; ++t)\n        for (int e = 0; e < E; ++e)\n            for (int j = 0; j < k; ++j)\n                if (idx_out[(size_t)t * k + j] == e) {"),
    ("bf16_ties_odd", "((cb >> 16) & 1u) == 0", "((cb >> 16) & 1u) == 1"),
    ("bf16_truncate", "if (dist < bestd ||", "if (step == 0 ||"),
    ("rmsnorm_no_eps", "double scale = 1.0 / sqrt(ss / d + eps);", "double scale = 1.0 / sqrt(ss / d);"),
    ("rmsnorm_sum_not_mean", "double scale = 1.0 / sqrt(ss / d + eps);", "double scale = 1.0 / sqrt(ss + eps);"),
    ("counts_off_by_one", "offsets[e + 1] = offsets[e] + counts[e];", "offsets[e + 1] = offsets[e] + counts[e] + (e == 0);"),
    ("second_slot_same_as_first", "if (taken)\n                continue;", "if (taken && j == 0)\n                continue;"),
    ("full_softmax_unnormalised", "g[j] = exp((double)l[chosen[j]] - l0) / zall;",
     "g[j] = exp((double)l[chosen[j]] - l0);"),
    ("full_softmax_over_kept", "zall += exp((double)l[e] - l0);", "zall += exp((double)l[e] - l0) * (e < 2);"),
    ("capacity_off_by_one", "taken[e] < capacity", "taken[e] <= capacity"),
    ("capacity_per_slot", "int e = idx[(size_t)t * k + j];\n            kept",
     "int e = j;\n            kept"),
    ("renorm_ignores_total", "g0[j] * total / kept_total", "g0[j] / kept_total"),
    ("dropped_row_kept_in_grouping", "if (!kept[(size_t)t * k + j]) {", "if (0) {"),
    # backward
    ("bwd_silu_prime_missing_term", "du[c] = dh * v[c] * (s + u[c] * s * (1.0 - s));",
     "du[c] = dh * v[c] * s;"),
    ("bwd_dv_uses_v", "dv[c] = dh * u[c] * s;", "dv[c] = dh * v[c] * s;"),
    ("bwd_softmax_not_centred", "DL[(size_t)t * k + j] = g[j] * (dg[j] - gdg);",
     "DL[(size_t)t * k + j] = g[j] * dg[j];"),
    ("bwd_dx_without_router_term", "DL[(size_t)t * k + j] * elem(Wg, (size_t)chosen[j] * d + i, dt);",
     "0.0 * elem(Wg, (size_t)chosen[j] * d + i, dt);"),
    ("bwd_dy_ungated", "dy[n] = g[j] * o;", "dy[n] = o;"),
    ("bwd_dW1_from_dv", "a1 += DU[s * ffn + c] * xi;", "a1 += DV[s * ffn + c] * xi;"),
    ("bwd_dW2_shifted", "a += DY[s * d + n] * H[s * ffn + c];",
     "a += DY[s * d + n] * H[s * ffn + (c + 1) % ffn];"),
    ("bwd_dx_w1_transposed", "acc += elem(W1[e], (size_t)c * d + i, dt) * du[c] +",
     "acc += elem(W1[e], (size_t)i * ffn + c, dt) * du[c] +"),
    ("bwd_dWg_sign", "acc += DL[s] * elem(x, (s / (size_t)k) * d + (size_t)i, dt);",
     "acc -= DL[s] * elem(x, (s / (size_t)k) * d + (size_t)i, dt);"),
    ("bwd_dh_without_w2", "dh += elem(W2[e], (size_t)n * ffn + c, dt) * dy[n];",
     "dh += dy[n];"),
]

RUNNER = r"""
import sys, traceback
sys.path[:0] = [{root!r}, {tests!r}]
import oracle, pins
o = oracle.load({lib!r})
failed = []
for p in pins.ALL:
    try:
        p(o)
    except Exception:
        failed.append(p.__name__)
print("FAILED:" + ",".join(failed))
sys.exit(1 if failed else 0)
"""


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_mutant(name, old, new, tmp_path):
    src = open(os.path.join(ROOT, "oracle", "moe_oracle.c")).read()
    assert src.count(old) == 1, f"mutation site for {name} not unique/present"
    mutated = tmp_path / "moe_oracle_mutant.c"
    mutated.write_text(src.replace(old, new))
    lib = str(tmp_path / "libmutant.so")
    oracle.build(str(mutated), lib)
    code = RUNNER.format(root=ROOT, tests=HERE, lib=lib)
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True,
                       timeout=300)
    assert r.returncode != 0, f"no pin caught mutant {name}: {r.stdout[-500:]} {r.stderr[-500:]}"
    assert "FAILED:" in r.stdout and r.stdout.strip().split("FAILED:")[-1], r.stdout
