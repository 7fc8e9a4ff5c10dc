"""Pins of the oracle's rotary step (YaRN frequencies, rotate-half application).

The pages show the rotary calls and the rope_scaling block of config.json (theta 50000, YaRN
factor 32 over 4096 original positions, beta_fast 1, beta_slow 1, mscale 1, mscale_all_dim
1) but not the function bodies; the oracle restates the published YaRN method.  Pins:
  - factor 1 reduces to plain rotary frequencies theta^(-2d/64), mscale ratio 1;
  - with the page's configuration the high-frequency dimensions (many rotations over the
    original context) keep the plain frequency and the low-frequency ones are divided by the
    factor, with the split where theta^(2d/64) * 2 pi * beta = 4096;
  - the mscale ratio m(s, a) / m(s, b) with m(s, k) = 0.1 k ln s + 1;
  - position 0 is the identity (query 0 of an empty cache against key 0);
  - a single active frequency pair gives closed-form scores between a query at position p
    and a key at position j (pins that queries rotate at past_len + i, new keys at their own
    position, cached keys are not rotated again, and the sign of the sine terms).
"""
import math

import numpy as np
import pytest
import torch

from oracle import oracle_rows, oracle_rows_rope, rotate, yarn
from mla_causal_attention_gb300.workloads import softmax_scale_192

PAGE = dict(theta=50000.0, factor=32.0, orig_max_pos=4096, beta_fast=1.0, beta_slow=1.0,
            mscale=1.0, mscale_all_dim=1.0)


def test_factor_one_is_plain_rotary():
    f, r = yarn(50000.0, 1.0, 4096, 32.0, 1.0, 1.0, 1.0)
    want = np.array([50000.0 ** (-2.0 * d / 64.0) for d in range(32)])
    np.testing.assert_allclose(f, want, rtol=1e-15)
    assert r == 1.0


def test_page_configuration_split():
    f, r = yarn(**PAGE)
    plain = np.array([50000.0 ** (-2.0 * d / 64.0) for d in range(32)])
    # number of rotations over the original context per dimension
    rotations = 4096 * plain / (2 * math.pi)
    keep = rotations > 1.0 + 1e-9
    # dimensions below the split keep the plain frequency, the others are interpolated
    assert keep[:19].all() and not keep[21:].any()
    np.testing.assert_allclose(f[:19], plain[:19], rtol=1e-15)
    np.testing.assert_allclose(f[21:], plain[21:] / 32.0, rtol=1e-15)
    assert r == 1.0


def test_mscale_ratio_closed_form():
    _, r = yarn(50000.0, 32.0, 4096, 1.0, 1.0, 2.0, 1.0)
    assert r == pytest.approx((0.2 * math.log(32) + 1) / (0.1 * math.log(32) + 1), rel=1e-15)


def _case(B, H, Tq, past, seed):
    g = torch.Generator("cpu").manual_seed(seed)
    Tk = past + Tq
    mk = lambda *s: torch.randn(*s, generator=g).to(torch.bfloat16)  # noqa: E731
    return dict(q_nope=mk(B, H, Tq, 128), q_pe=mk(B, H, Tq, 64), k_nope=mk(B, H, Tk, 128),
                k_pe_shared=mk(B, Tk, 64), v=mk(B, H, Tk, 128))


def test_position_zero_is_identity():
    d = _case(1, 2, 1, 0, seed=1)
    f, r = yarn(**PAGE)
    args = (d["q_nope"], d["q_pe"], d["k_nope"], d["k_pe_shared"], d["v"], None, 0,
            softmax_scale_192())
    np.testing.assert_allclose(oracle_rows_rope(*args, f, r), oracle_rows(*args), atol=0)


@pytest.mark.parametrize("dim", [3, 25])   # one extrapolated, one interpolated frequency
def test_single_frequency_closed_form(dim):
    """Only the pair (dim, dim + 32) is non-zero.  A rotation by angle t maps (x1, x2) to
    (x1 cos t - x2 sin t, x2 cos t + x1 sin t), so a query at position p against a new key at
    position j scores (u1 w1 + u2 w2) cos t + (u2 w1 - u1 w2) sin t with t = (j - p) f, and
    against a cached (already rotated) key wc scores the same form with t = -p f."""
    past, Tq = 5, 2
    d = _case(1, 1, Tq, past, seed=2)
    for k in ("q_nope", "q_pe", "k_nope", "k_pe_shared"):
        d[k].zero_()
    u1, u2 = 2.0, -0.75    # raw query rotary pair
    w1, w2 = 1.5, 0.5      # raw new keys
    c1, c2 = -0.5, 1.25    # cached keys, stored rotated
    d["q_pe"][0, 0, :, dim] = u1
    d["q_pe"][0, 0, :, dim + 32] = u2
    d["k_pe_shared"][0, past:, dim] = w1
    d["k_pe_shared"][0, past:, dim + 32] = w2
    d["k_pe_shared"][0, :past, dim] = c1
    d["k_pe_shared"][0, :past, dim + 32] = c2
    f, r = yarn(**PAGE)
    sc = float(np.float32(softmax_scale_192()))
    out = oracle_rows_rope(d["q_nope"], d["q_pe"], d["k_nope"], d["k_pe_shared"], d["v"], None,
                           past, softmax_scale_192(), f, r)
    v = d["v"].double().numpy()[0, 0]

    def pair(x1, x2, y1, y2, t):
        return (x1 * y1 + x2 * y2) * math.cos(t) + (x2 * y1 - x1 * y2) * math.sin(t)

    for i in range(Tq):
        pos = past + i
        s = [pair(u1, u2, c1, c2, -pos * f[dim]) * sc for _ in range(past)]
        s += [pair(u1, u2, w1, w2, (j - pos) * f[dim]) * sc for j in range(past, past + Tq)]
        vis = [j for j in range(past + Tq) if j <= pos]
        e = np.array([math.exp(s[j]) for j in vis])
        want = (e[:, None] * v[vis]).sum(0) / e.sum()
        np.testing.assert_allclose(out[i], want, rtol=0, atol=1e-12)


@pytest.mark.parametrize("dim", [0, 7, 19, 20, 31])
def test_rotate_unit_vectors(dim):
    """The rotation alone on unit vectors: e_d at position p goes to cos(p f_d) e_d +
    sin(p f_d) e_{d+32}, and e_{d+32} to -sin(p f_d) e_d + cos(p f_d) e_{d+32} (a
    counter-clockwise turn of the pair by the angle p f_d), times the mscale ratio."""
    f, _ = yarn(**PAGE)
    x = torch.zeros(2, 64, dtype=torch.bfloat16)
    x[0, dim] = 1.0
    x[1, dim + 32] = 1.0
    for p in (1, 4095, 131071):
        for ratio in (1.0, 1.25):
            y = rotate(x, p, f, ratio)
            a = p * f[dim]
            want = np.zeros((2, 64))
            want[0, dim], want[0, dim + 32] = math.cos(a), math.sin(a)
            want[1, dim], want[1, dim + 32] = -math.sin(a), math.cos(a)
            np.testing.assert_allclose(y, want * ratio, rtol=0, atol=1e-15)


def test_rotate_is_the_step_inside_attention():
    """Rotating the query and the new keys with rotate() at positions past_len + t, rounding
    them to bf16 and running the rotation-free oracle matches oracle_rows_rope up to that
    rounding (about 1e-3 here); a position off by one in either moves the output by 0.1."""
    past, Tq = 7, 5
    d = _case(1, 2, Tq, past, seed=5)
    f, r = yarn(**PAGE)
    sc = softmax_scale_192()
    want = oracle_rows_rope(d["q_nope"], d["q_pe"], d["k_nope"], d["k_pe_shared"], d["v"],
                            None, past, sc, f, r)
    pos = np.arange(Tq) + past
    q_rot = torch.from_numpy(rotate(d["q_pe"], pos[None, None, :], f, r)).to(torch.bfloat16)
    k_rot = d["k_pe_shared"].clone()
    k_rot[:, past:] = torch.from_numpy(
        rotate(d["k_pe_shared"][:, past:], pos[None, :], f, r)).to(torch.bfloat16)
    got = oracle_rows(d["q_nope"], q_rot, d["k_nope"], k_rot, d["v"], None, past, sc)
    np.testing.assert_allclose(got, want, rtol=0, atol=1e-2)
