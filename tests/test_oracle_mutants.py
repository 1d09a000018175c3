"""Plant plausible mistakes in copies of the oracle; every one must fail some pin.

Each mutant is a one-site textual edit of oracle.c (asserted to match exactly
once), compiled with gcc into a temporary library.  Nothing here touches a GPU.
"""
import os
import subprocess
import tempfile

import pytest

import oracle
import _pins

SRC = os.path.join(os.path.dirname(os.path.abspath(oracle.__file__)), "oracle.c")

# (name, original text, mutated text)
MUTANTS = [
    ("lse_sign", "c->lse[((size_t)b * c->Hq + h) * c->S + s] = m + log(den)",
     "c->lse[((size_t)b * c->Hq + h) * c->S + s] = -m + log(den)"),
    ("gqa_interleaved", "int G = c->Hq / c->Hkv, g = h / G;", "int G = c->Hq / c->Hkv, g = h % c->Hkv;"),
    ("prefix_off_by_one", "    if (j < L)\n", "    if (j <= L)\n"),
    ("dropped_scale", "x[j] = c->scale * dot;", "x[j] = dot;"),
    ("value_uses_key", "const uint16_t *vr = key_row(c, c->v_ctx, c->v_blk, b, g, j);",
     "const uint16_t *vr = key_row(c, c->k_ctx, c->k_blk, b, g, j);"),
    ("dropped_block_keys", "(c->keys == KEYS_BLOCK ? c->S : L + c->S)",
     "(c->keys == KEYS_BLOCK ? c->S : L + 1)"),
    ("q_layout_transposed", "bf16_to_double(c->q[qi + e])",
     "bf16_to_double(c->q[(((size_t)b * c->Hq + h) * c->S + s) * d + e])"),
    ("dropped_normaliser", "* (acc[e] / den);", "* (acc[e]);"),
    ("temperature_multiplies", "- best) / c->temperature);", "- best) * c->temperature);"),
    ("argmax_last_tie", "if (l > best) { best = l; arg = v; }", "if (l >= best) { best = l; arg = v; }"),
    ("threshold_strict", "if (force_commit_all || cf >= threshold) {",
     "if (force_commit_all || cf > threshold) {"),
    ("fallback_tie_high", "if (best < 0 || cf > (float)conf[base + best])",
     "if (best < 0 || cf >= (float)conf[base + best])"),
    ("no_remask", "tokens[base + s] = mask_token_id;", "(void)mask_token_id;"),
    ("no_fallback", "if (n_masked > 0 && n_pass == 0) {", "if (0) {"),
    ("force_ignored", "if (force_commit_all || cf >= threshold) {", "if (cf >= threshold) {"),
    ("conf_is_sum", "c->conf[row] = 1.0 / sum;", "c->conf[row] = sum;"),
]


def test_mutant_sites_exist():
    src = open(SRC).read()
    for name, old, _ in MUTANTS:
        assert src.count(old) == 1, name


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(name, old, new):
    src = open(SRC).read()
    assert src.count(old) == 1
    with tempfile.TemporaryDirectory() as tmp:
        c_path = os.path.join(tmp, "mutant.c")
        so_path = os.path.join(tmp, "libmutant.so")
        with open(c_path, "w") as f:
            f.write(src.replace(old, new))
        subprocess.run(["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-pthread", c_path, "-o",
                        so_path, "-lm"], check=True, capture_output=True)
        lib = oracle.load(so_path)
        failures = []
        for check in _pins.ALL_CHECKS:
            try:
                check(lib)
            except AssertionError:
                failures.append(check.__name__)
            except (ValueError, FloatingPointError):
                failures.append(check.__name__)
        assert failures, f"mutant {name} passed every pin"
