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


# Mistakes in the rotary step, checked against the rotary pins.
ROPE_MUTANTS = {
    "rope_query_position_ignores_past": (
        "rotate64(q + D_NOPE, raw, (double)(J->past_len + i),",
        "rotate64(q + D_NOPE, raw, (double)(i),"),
    "rope_cached_keys_rotated_again": ("if (J->rope_inv_freq && j >= J->past_len) {",
                                       "if (J->rope_inv_freq) {"),
    "rope_sine_sign": ("y[d] = x[d] * c - x[d + 32] * sn;", "y[d] = x[d] * c + x[d + 32] * sn;"),
    "rope_ramp_inverted": ("inv_freq[d] = inter * ramp + extra * (1.0 - ramp);",
                           "inv_freq[d] = extra * ramp + inter * (1.0 - ramp);"),
    "rope_pairs_adjacent": ("y[d + 32] = x[d + 32] * c + x[d] * sn;",
                            "y[d + 32] = x[d + 32] * c + x[(d + 1) & 31] * sn;"),
}


# Mistakes in the 2D padding mask, checked against the mask pins.
MASK_MUTANTS = {
    "mask_ignored": ("(!J->key_mask || J->key_mask[b * J->Tk + j] != 0)", "1"),
    "mask_inverted": ("J->key_mask[b * J->Tk + j] != 0", "J->key_mask[b * J->Tk + j] == 0"),
    "mask_wrong_sequence": ("J->key_mask[b * J->Tk + j]", "J->key_mask[j]"),
    "hidden_keys_dropped": ("sj += visible ? 0.0 : MASK_MIN_BF16;",
                            "sj = visible ? sj : -INFINITY;"),
}


# Mistakes in the latent-cache rows, checked against the latent pins.
LATENT_MUTANTS = {
    "latent_key_value_swapped": ("const uint16_t* wk = J->w_kvb + (h * 256) * D_LAT;",
                                 "const uint16_t* wk = J->w_kvb + (h * 256 + 128) * D_LAT;"),
    "latent_head_ignored": ("const uint16_t* wv = J->w_kvb + (h * 256 + 128) * D_LAT;",
                            "const uint16_t* wv = J->w_kvb + (128) * D_LAT;"),
    "latent_weight_transposed": ("kn += bf16_to_double(wk[e * D_LAT + d]) * bf16_to_double(c[d]);",
                                 "kn += bf16_to_double(wk[d * 128 + e]) * bf16_to_double(c[d]);"),
    "latent_rope_dropped": ("acc += q[D_NOPE + d] * bf16_to_double(kr[d]); /* shared rotary key */",
                            "acc += 0.0; /* shared rotary key */"),
}

# Mistakes in the output projection, checked against its pins.
OPROJ_MUTANTS = {
    "oproj_weight_transposed": ("const uint16_t* wr = J->w + n * J->K; /* row n of the weight */",
                                "const uint16_t* wr = J->w + n; /* row n of the weight */"),
    "oproj_head_order": ("for (int64_t d = 0; d < D_V; ++d) x[h * D_V + d] = bf16_to_double(src[d]);",
                         "for (int64_t d = 0; d < D_V; ++d) x[d * J->H + h] = bf16_to_double(src[d]);"),
    "oproj_time_ignored": ("const uint16_t* src = J->attn + ((b * J->H + h) * J->T + i) * D_V;",
                           "const uint16_t* src = J->attn + ((b * J->H + h) * J->T) * D_V;"),
    "oproj_last_head_dropped": ("for (int64_t h = 0; h < J->H; ++h) { /* concatenated head outputs */",
                                "for (int64_t h = 0; h < J->H; ++h) { if (h == J->H - 1) { for (int64_t d = 0; d < D_V; ++d) x[h * D_V + d] = 0.0; continue; }"),
}


def _run_pins(name, old, new, tmp_path, pin_file):
    src = open(SRC).read()
    assert old in src, f"mutation site for {name} not found"
    mut = tmp_path / "mut.c"
    mut.write_text(src.replace(old, new))
    lib = tmp_path / "libmut.so"
    subprocess.run(["gcc", "-O2", "-ffp-contract=off", "-fPIC", "-shared", "-pthread", "-o",
                    str(lib), str(mut), "-lm"], check=True)
    env = dict(os.environ, MLA_ORACLE_LIB=str(lib))
    r = subprocess.run([sys.executable, "-m", "pytest", os.path.join(ROOT, "tests", pin_file),
                        "-q", "-x", "-p", "no:cacheprovider"],
                       capture_output=True, text=True, env=env, cwd=ROOT, timeout=300)
    assert r.returncode == 1, f"mutant {name} survived the pins:\n{r.stdout[-2000:]}"


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_kill_mutant(name, tmp_path):
    old, new = MUTANTS[name]
    _run_pins(name, old, new, tmp_path, "test_oracle.py")


@pytest.mark.parametrize("name", sorted(ROPE_MUTANTS))
def test_rope_pins_kill_mutant(name, tmp_path):
    old, new = ROPE_MUTANTS[name]
    _run_pins(name, old, new, tmp_path, "test_oracle_rope.py")


@pytest.mark.parametrize("name", sorted(MASK_MUTANTS))
def test_mask_pins_kill_mutant(name, tmp_path):
    old, new = MASK_MUTANTS[name]
    _run_pins(name, old, new, tmp_path, "test_oracle_mask.py")


@pytest.mark.parametrize("name", sorted(LATENT_MUTANTS))
def test_latent_pins_kill_mutant(name, tmp_path):
    old, new = LATENT_MUTANTS[name]
    _run_pins(name, old, new, tmp_path, "test_oracle_latent.py")


@pytest.mark.parametrize("name", sorted(OPROJ_MUTANTS))
def test_oproj_pins_kill_mutant(name, tmp_path):
    old, new = OPROJ_MUTANTS[name]
    _run_pins(name, old, new, tmp_path, "test_oracle_oproj.py")
