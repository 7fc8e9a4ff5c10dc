"""The oracle's pins must fail on plausible planted mistakes.

Each case copies mla_oracle.c to a temporary directory, plants one mistake there (the
committed source is never touched), builds it, and runs test_oracle.py against that build
through MLA_ORACLE_LIB.  A mutant that passes every pin means the pins are too weak.
"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "mla_oracle.c")

MUTANTS = {
    "drop_rope_term": ("acc += q[D_NOPE + d] * bf16_to_double(kr[d]);", "acc += 0.0;"),
    "drop_nope_term": ("acc += q[d] * bf16_to_double(kn[d]);", "acc += 0.0;"),
    "causal_off_by_one": ("(j <= i + J->past_len)", "(j < i + J->past_len)"),
    "causal_ignores_past": ("(j <= i + J->past_len)", "(j <= i)"),
    "padding_off_by_one": ("(j < kvl)", "(j <= kvl)"),
    "rope_key_per_head": ("J->k_pe + (b * J->Tk + j) * D_ROPE",
                          "J->k_pe + ((bh % J->B) * J->Tk + j) * D_ROPE"),
    "softmax_sign": ("s[j] = exp(s[j] - m);", "s[j] = exp(m - s[j]);"),
    "scale_dropped": ("double sj = acc * scale_used;", "double sj = acc;"),
    "no_normalisation": ("s[j] = s[j] / denom;", "s[j] = s[j] * 1.0;"),
    "values_reversed": ("J->v + (bh * J->Tk + j) * D_V",
                        "J->v + (bh * J->Tk + (J->Tk - 1 - j)) * D_V"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_kill_mutant(name, tmp_path):
    src = open(SRC).read()
    old, new = MUTANTS[name]
    assert old in src, f"mutation site for {name} not found"
    mut = tmp_path / "mut.c"
    mut.write_text(src.replace(old, new))
    lib = tmp_path / "libmut.so"
    subprocess.run(["gcc", "-O2", "-ffp-contract=off", "-fPIC", "-shared", "-pthread", "-o",
                    str(lib), str(mut), "-lm"], check=True)
    env = dict(os.environ, MLA_ORACLE_LIB=str(lib))
    r = subprocess.run([sys.executable, "-m", "pytest", os.path.join(ROOT, "tests",
                        "test_oracle.py"), "-q", "-x", "-p", "no:cacheprovider"],
                       capture_output=True, text=True, env=env, cwd=ROOT, timeout=300)
    assert r.returncode == 1, f"mutant {name} survived the pins:\n{r.stdout[-2000:]}"
