"""Planted mistakes in a copy of the oracle must each fail a pin (CPU only).

Every mutation below is a plausible slip in the oracle's C source:
- in the forward pass: a reordered, unfused or unblocked logit chain, the wrong
  tie-break, a dropped renormalisation, a sign error in SiLU, swapped gate/up
  branches or pre-activations, a dropped routing weight, truncating instead of
  rounding, a transposed weight, an unstable grouping;
- in Token Rounding: a wrong rounding rule, a wrong order in the second sort or
  a dropped renormalisation;
- in the backward pass: a wrong SiLU derivative, a dropped routing weight or
  renormalisation term, or the wrong weight in dX.
The test copies the oracle into a temporary directory, applies one mutation,
rebuilds it there and runs the pin suites against the copy; they have to fail.
"""
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

MUTATIONS = [
    ("unfused_logits", "blk[e] = fmaf(xj, w[e], blk[e]);", "blk[e] = blk[e] + xj * w[e];"),
    ("descending_j", "for (int j = j0; j < j1; ++j) {\n            float xj",
     "for (int j = j1 - 1; j >= j0; --j) {\n            float xj"),
    ("logits_unblocked", "#define LOGIT_BLOCK 1024", "#define LOGIT_BLOCK (1 << 30)"),
    ("logits_blocked_for_every_E", "#define LOGIT_FEW_EXPERTS 32", "#define LOGIT_FEW_EXPERTS (1 << 30)"),
    ("logit_blocks_not_restarted", "for (int e = 0; e < E; ++e) blk[e] = 0.0f;", ""),
    ("ties_to_high_index", "return (a->e > b->e) - (a->e < b->e);",
     "return (a->e < b->e) - (a->e > b->e);"),
    ("no_renorm", "renorm ? p / kept : p", "p"),
    ("silu_sign", "a / (1.0 + exp(-a))", "a / (1.0 + exp(a))"),
    ("gate_up_swapped", "silu(a1[j]) * a3[j]", "silu(a3[j]) * a1[j]"),
    ("combine_drops_k0", "for (int k = 0; k < K; ++k) y = y + Z[", "for (int k = 1; k < K; ++k) y = y + Z["),
    ("weight_dropped", "z[c] = w * z[c];", "z[c] = z[c];"),
    ("bf16_truncates", "nearbyint(ldexp(a, -e_ulp))", "floor(ldexp(a, -e_ulp))"),
    ("bias_sign", "acc[e] = acc[e] + bias[e];", "acc[e] = acc[e] - bias[e];"),
    ("tile_rows_unclipped", "(c - r < M) ? (c - r) : M", "M"),
    ("denominator_short", "for (int e = 0; e < E; ++e) denom +=", "for (int e = 0; e < E - 1; ++e) denom +="),
    ("w2_transposed", "const uint16_t *w2 = W2e + (int64_t)j * d;", "const uint16_t *w2 = W2e + (int64_t)j;"),
    ("grouping_reversed", "for (int64_t t = 0; t < T; ++t)\n        for (int k = 0; k < K; ++k) {\n            int32_t slot",
     "for (int64_t t = T - 1; t >= 0; --t)\n        for (int k = 0; k < K; ++k) {\n            int32_t slot"),
    ("gather_ignores_perm", "const uint16_t *x = X + (int64_t)perm_token[p] * d;",
     "const uint16_t *x = X + (int64_t)p * d;"),
    ("pre_activations_swapped", "A1 + (int64_t)p * n, A3 + (int64_t)p * n, h);",
     "A3 + (int64_t)p * n, A1 + (int64_t)p * n, h);"),
    # Token Rounding
    ("tr_always_round_down", "(int64_t)M * ((f[e] + M / 2) / M);", "(int64_t)M * (f[e] / M);"),
    ("tr_always_round_up", "(int64_t)M * ((f[e] + M / 2) / M);", "(int64_t)M * ((f[e] + M - 1) / M);"),
    ("tr_halves_down", "(int64_t)M * ((f[e] + M / 2) / M);", "(int64_t)M * ((f[e] + (M - 1) / 2) / M);"),
    ("tr_no_cap_at_T", "if (c > T) c = (int64_t)M * (f[e] / M);", ""),
    ("tr_members_not_first", "return a->member ? -1 : 1;", "return a->member ? 1 : -1;"),
    ("tr_low_scores_first", "if (a->v > b->v) return -1;\n    if (a->v < b->v) return 1;\n    return (a->t",
     "if (a->v < b->v) return -1;\n    if (a->v > b->v) return 1;\n    return (a->t"),
    ("tr_ties_to_high_token", "return (a->t > b->t) - (a->t < b->t);", "return (a->t < b->t) - (a->t > b->t);"),
    ("tr_renorm_ignored", "renorm ? pe / kept : pe", "pe"),
    ("tr_row_order_descending_t", "for (int e = 0; e < E; ++e)\n        for (int64_t t = 0; t < T; ++t) {\n            if (keep",
     "for (int e = 0; e < E; ++e)\n        for (int64_t t = T - 1; t >= 0; --t) {\n            if (keep"),
    ("combine_rows_skips_row0", "if (r >= 0) y = y + Z[", "if (r > 0) y = y + Z["),
    # backward
    ("bwd_silu_derivative", "s * (1.0 + a1[i] * (1.0 - s))", "s * (1.0 + a1[i] * s)"),
    ("bwd_dh_unweighted", "dh[i] = w[k] * gw;", "dh[i] = gw;"),
    # backward, per row
    ("bwd_rows_ds_drops_a3", "ds += silu(u) * v * q;", "ds += silu(u) * q;"),
    ("bwd_rows_dxg_w3_for_w1", "acc += r1[i] * W1e[(int64_t)j * n + i] + r3[i] * W3e",
     "acc += r1[i] * W3e[(int64_t)j * n + i] + r3[i] * W3e"),
    ("bwd_rows_renorm_mean_dropped", "dl[e] += renorm ? (s - sw) / kept : s;",
     "dl[e] += renorm ? s / kept : s;"),
    ("bwd_dw2_unweighted", "+= h * w[k] * g[c];", "+= h * g[c];"),
    ("bwd_router_renorm_term_dropped", "(dw[k] - wdw) / kept", "dw[k] / kept"),
    ("bwd_dx_through_w1_twice", "da3 * W3e[(int64_t)j * n + i]", "da3 * W1e[(int64_t)j * n + i]"),
]

PIN_FILES = ["test_oracle_pins.py", "test_oracle_rounding.py", "test_oracle_backward.py"]


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistake_fails_a_pin(tmp_path, name, old, new):
    src = open(os.path.join(ROOT, "oracle", "moe_oracle.c")).read()
    assert src.count(old) >= 1, "mutation site not found: " + name
    dst = tmp_path / "oracle"
    shutil.copytree(os.path.join(ROOT, "oracle"), dst,
                    ignore=shutil.ignore_patterns("_build", "__pycache__"))
    (dst / "moe_oracle.c").write_text(src.replace(old, new))
    env = dict(os.environ, PYTHONPATH=f"{tmp_path}{os.pathsep}{ROOT}")
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                        *[os.path.join(ROOT, "tests", f) for f in PIN_FILES]],
                       env=env, capture_output=True, text=True, cwd=str(tmp_path), timeout=600)
    assert r.returncode != 0, f"mutation {name} passed every pin:\n{r.stdout[-2000:]}"
