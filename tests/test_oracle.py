"""Pins of the fp64 CPU oracle against facts fixed by the pages and by mathematics.

Each test is chosen so that a plausible mistake in the oracle fails it:
  - a dropped score term (no-rope or rope part)      -> two-key closed forms, SDPA
  - a wrong sign / swapped weights                   -> two-key closed forms
  - an off-by-one or wrong offset in the mask        -> equal-score means, SDPA
  - the rotary key indexed per head, not shared      -> shared-key test, SDPA
  - a transposed operand / wrong row stride          -> SDPA with Tq != Tk, H > 1, B > 1
  - a wrong normalisation                            -> weight sums, all-ones values
None of these tests needs a GPU.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import oracle_rows, round_bf16
from mla_causal_attention_gb300.inputs import make_inputs
from mla_causal_attention_gb300.workloads import WORKLOADS, Workload, softmax_scale_192

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
MASK_MIN = torch.finfo(torch.bfloat16).min  # the dtype-min the 4D mask holds


def rand_case(B, H, Tq, past, seed, kv_len=None, scale=1.0):
    g = torch.Generator("cpu").manual_seed(seed)
    Tk = past + Tq
    mk = lambda *s: (torch.randn(*s, generator=g) * scale).to(torch.bfloat16)  # noqa: E731
    d = dict(q_nope=mk(B, H, Tq, 128), q_pe=mk(B, H, Tq, 64), k_nope=mk(B, H, Tk, 128),
             k_pe_shared=mk(B, Tk, 64), v=mk(B, H, Tk, 128))
    d["kv_len"] = (torch.full((B,), Tk, dtype=torch.int32) if kv_len is None
                   else torch.tensor(kv_len, dtype=torch.int32))
    d["past_len"] = past
    return d


def run(d, scale=softmax_scale_192(), **kw):
    B, H, Tq = d["q_nope"].shape[:3]
    o = oracle_rows(d["q_nope"], d["q_pe"], d["k_nope"], d["k_pe_shared"], d["v"], d["kv_len"],
                    d["past_len"], scale, **kw)
    if kw.get("return_wsum"):
        return o[0].reshape(B, H, Tq, 128), o[1].reshape(B, H, Tq)
    return o.reshape(B, H, Tq, 128)


def f64(t):
    return t.to(torch.float64).numpy()


def visible_count(i, past, kvl):
    return min(i + past + 1, kvl)


# --- P1: weights of every row sum to one -------------------------------------------------
@pytest.mark.parametrize("B,H,Tq,past,kv", [(1, 2, 7, 0, None), (2, 3, 5, 4, [9, 3]),
                                            (2, 1, 1, 30, [31, 12])])
def test_weight_rows_sum_to_one(B, H, Tq, past, kv):
    d = rand_case(B, H, Tq, past, seed=1, kv_len=kv, scale=3.0)
    _, wsum = run(d, return_wsum=True)
    assert np.all(np.abs(wsum - 1.0) <= 1e-12)
    d["v"] = torch.ones_like(d["v"])  # all-ones values: every output element is sum(w) = 1
    out = run(d)
    assert np.all(np.abs(out - 1.0) <= 1e-12)


# --- P2: a single visible key returns that key's value row exactly -------------------------
def test_single_visible_key_returns_its_value():
    d = rand_case(2, 3, 6, 0, seed=2)
    out = run(d)
    # with no cached prefix, query 0 sees only key 0
    assert np.array_equal(out[:, :, 0, :], f64(d["v"][:, :, 0, :]))


def test_kv_len_one_returns_first_value_for_every_query():
    d = rand_case(2, 2, 4, 5, seed=3, kv_len=[1, 1])
    out = run(d)
    for i in range(4):
        assert np.array_equal(out[:, :, i, :], f64(d["v"][:, :, 0, :]))


# --- P3: equal scores give the mean of the visible value rows (mask offsets) ---------------
@pytest.mark.parametrize("past,kv", [(0, None), (3, None), (6, [8, 2]), (2, [4, 7])])
def test_equal_scores_average_visible_values(past, kv):
    B, H, Tq = 2, 2, 5
    d = rand_case(B, H, Tq, past, seed=4, kv_len=kv)
    d["q_nope"].zero_()
    d["q_pe"].zero_()
    out = run(d)
    kvl = d["kv_len"].numpy()
    v = f64(d["v"])
    for b in range(B):
        for i in range(Tq):
            n = visible_count(i, past, int(kvl[b]))
            np.testing.assert_allclose(out[b, :, i, :], v[b, :, :n, :].mean(axis=1),
                                       rtol=0, atol=1e-13)


# --- P4: keys the mask hides do not change the output at all --------------------------------
def test_hidden_keys_do_not_matter():
    B, H, Tq, past = 2, 2, 6, 3
    kv = [7, 5]
    d = rand_case(B, H, Tq, past, seed=5, kv_len=kv)
    base = run(d)
    Tk = past + Tq
    # Poison every key/value row at or beyond kv_len[b] with finite huge values.
    for b in range(B):
        d["k_nope"][b, :, kv[b]:, :] = 1e30
        d["v"][b, :, kv[b]:, :] = -1e30
        d["k_pe_shared"][b, kv[b]:, :] = 1e30
    assert np.array_equal(run(d), base)
    # Causal part: changing key rows after position i+past must leave row i unchanged.
    d2 = rand_case(1, 1, 5, 0, seed=6)
    ref = run(d2)
    d2["k_nope"][0, 0, 3:, :] = 7.0
    d2["v"][0, 0, 3:, :] = 9.0
    out = run(d2)
    assert np.array_equal(out[0, 0, :3], ref[0, 0, :3])
    assert not np.array_equal(out[0, 0, 3:], ref[0, 0, 3:])
    assert Tk == 9


# --- Two-key closed forms: w0 = 1/(1 + exp(s1 - s0)) ----------------------------------------
def _two_key_case(part):
    """One query (past_len=1, Tq=1, Tk=2) with the score signal in one part only."""
    d = rand_case(1, 2, 1, 1, seed=7)
    for k in ("q_nope", "q_pe", "k_nope", "k_pe_shared"):
        d[k].zero_()
    if part == "nope":
        d["q_nope"][0, :, 0, 5] = 2.0
        d["q_nope"][0, 1, 0, 5] = -1.5  # head 1 differs
        d["k_nope"][0, :, 0, 5] = 1.0
        d["k_nope"][0, :, 1, 5] = 3.0
    else:  # rope: the key's rotary part is one row per sequence, shared by both heads
        d["q_pe"][0, 0, 0, 17] = 2.0
        d["q_pe"][0, 1, 0, 17] = -1.5
        d["k_pe_shared"][0, 0, 17] = 1.0
        d["k_pe_shared"][0, 1, 17] = 3.0
    return d


@pytest.mark.parametrize("part", ["nope", "rope"])
@pytest.mark.parametrize("scale", [0.25, softmax_scale_192()])
def test_two_key_closed_form(part, scale):
    d = _two_key_case(part)
    out = run(d, scale=scale)
    v = f64(d["v"])
    sc = float(np.float32(scale))
    for h, qv in ((0, 2.0), (1, -1.5)):
        s0, s1 = qv * 1.0 * sc, qv * 3.0 * sc
        w0 = 1.0 / (1.0 + math.exp(s1 - s0))
        want = w0 * v[0, h, 0] + (1.0 - w0) * v[0, h, 1]
        np.testing.assert_allclose(out[0, h, 0], want, rtol=0, atol=1e-14)


def test_rotary_key_is_shared_across_heads():
    d = _two_key_case("rope")
    d["q_pe"][0, 1, 0, 17] = 2.0  # both heads now ask the same question of the shared key
    out = run(d)
    v = f64(d["v"])
    # identical weights in both heads: out[h] = w0 v[h,0] + w1 v[h,1] with the same w0
    w0 = (out[0, 0, 0] - v[0, 0, 1]) / (v[0, 0, 0] - v[0, 0, 1])
    w0b = (out[0, 1, 0] - v[0, 1, 1]) / (v[0, 1, 0] - v[0, 1, 1])
    np.testing.assert_allclose(w0, w0b, rtol=0, atol=1e-9)


# --- Library special case: torch SDPA in float64 with the explicit additive mask ------------
@pytest.mark.parametrize("B,H,Tq,past,kv", [(2, 3, 5, 0, None), (2, 2, 4, 7, [11, 6]),
                                            (1, 4, 1, 9, [5]), (3, 1, 6, 2, [8, 1, 4])])
def test_matches_torch_sdpa_float64(B, H, Tq, past, kv):
    d = rand_case(B, H, Tq, past, seed=8, kv_len=kv, scale=2.0)
    scale = softmax_scale_192()
    out = run(d, scale=scale)
    Tk = past + Tq
    q = torch.cat([d["q_nope"], d["q_pe"]], dim=-1).double()
    kpe = d["k_pe_shared"][:, None, :, :].expand(B, H, Tk, 64)
    k = torch.cat([d["k_nope"], kpe], dim=-1).double()
    v = d["v"].double()
    mask = torch.zeros(B, 1, Tq, Tk, dtype=torch.float64)
    for b in range(B):
        for i in range(Tq):
            for j in range(Tk):
                if j > i + past or j >= int(d["kv_len"][b]):
                    mask[b, 0, i, j] = MASK_MIN
    ref = torch.nn.functional.scaled_dot_product_attention(
        q, k, v, attn_mask=mask, scale=float(np.float32(scale)))
    np.testing.assert_allclose(out, ref.numpy(), rtol=0, atol=1e-12)


# --- Brute force on tiny inputs: a pure-Python loop with exact-sum dot products -------------
def test_bruteforce_python_loop():
    B, H, Tq, past, kv = 2, 2, 3, 2, [4, 5]
    d = rand_case(B, H, Tq, past, seed=9, kv_len=kv)
    sc = float(np.float32(0.3))
    out = run(d, scale=0.3)
    qn, qr, kn, kr, v = (d[k].double().tolist() for k in
                         ("q_nope", "q_pe", "k_nope", "k_pe_shared", "v"))
    for b in range(B):
        for h in range(H):
            for i in range(Tq):
                keys = [j for j in range(past + Tq) if j <= i + past and j < kv[b]]
                s = {j: math.fsum([a * c for a, c in zip(qn[b][h][i] + qr[b][h][i],
                                                         kn[b][h][j] + kr[b][j])]) * sc
                     for j in keys}
                top = max(s.values())
                e = {j: math.exp(s[j] - top) for j in keys}
                z = math.fsum(e.values())
                for dd in range(128):
                    want = math.fsum(e[j] / z * v[b][h][j][dd] for j in keys)
                    assert abs(out[b, h, i, dd] - want) <= 1e-12


# --- Shapes printed on the pages ------------------------------------------------------------
def test_workloads_match_printed_shapes():
    g = json.load(open(os.path.join(GOLDEN, "kimi_k2_attention_shapes.json")))
    wl = WORKLOADS["decode_p1000"]
    assert (wl.H, 1, wl.Tk) == tuple(g["decode_p1000_scores_shape"][1:])
    assert wl.past_len == g["decode_p1000_cached_length"] and wl.Tq == 1
    for w in WORKLOADS.values():
        assert w.H == g["num_attention_heads"] == g["num_key_value_heads"]
    assert (g["qk_nope_head_dim"], g["qk_rope_head_dim"], g["v_head_dim"]) == (128, 64, 128)
    assert g["attention_dropout"] == 0.0  # dropout is the identity in this path
    inp = make_inputs(WORKLOADS["tiny_prefill"], seed=0)
    assert tuple(inp["v"].shape[1:]) == (64, 16, 128)
    # the latent width and the output projection's width, without bias
    from mla_causal_attention_gb300.workloads import D_LAT
    assert D_LAT == g["kv_lora_rank"]
    assert g["attention_bias"] is False
    import importlib.util
    spec = importlib.util.spec_from_file_location(
        "bench", os.path.join(os.path.dirname(GOLDEN), os.pardir, "bench.py"))
    bench = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(bench)
    for c in bench.OPROJ_WORKLOADS.values():
        assert c["N"] == g["hidden_size"] and c["H"] == g["num_attention_heads"]


def test_oracle_rejects_bad_arguments():
    d = rand_case(1, 1, 2, 0, seed=10, kv_len=[0])
    with pytest.raises(ValueError):
        run(d)
    d = rand_case(1, 1, 2, 0, seed=10, kv_len=[3])
    with pytest.raises(ValueError):
        run(d)


# --- The eager-emulation diagnostic ---------------------------------------------------------
def test_round_bf16_matches_torch_cast():
    g = torch.Generator("cpu").manual_seed(11)
    x = torch.cat([torch.randn(4000, generator=g, dtype=torch.float64) * 10,
                   torch.tensor([1.0 + 2**-8, 1.0 + 3 * 2**-8, -2.5, 0.0, 65504.0])])
    want = x.to(torch.float32).to(torch.bfloat16).to(torch.float64)
    got = torch.tensor([round_bf16(float(a)) for a in x], dtype=torch.float64)
    assert torch.equal(got, want)


def test_eager_mode_is_close_but_not_exact():
    d = rand_case(1, 2, 8, 4, seed=12)
    exact = run(d)
    eager = run(d, mode="eager")
    err = np.abs(exact - eager)
    assert err.max() < 2e-2 and err.max() > 0.0


def test_oracle_rows_subset_matches_full():
    d = rand_case(2, 2, 5, 3, seed=13, kv_len=[8, 6])
    full = run(d).reshape(-1, 128)
    rows = [0, 7, 19, 3]
    sub = oracle_rows(d["q_nope"], d["q_pe"], d["k_nope"], d["k_pe_shared"], d["v"],
                      d["kv_len"], d["past_len"], softmax_scale_192(), rows=rows)
    assert np.array_equal(sub, full[rows])


def test_ragged_workload_kv_len_range():
    wl = Workload("r", 3, 2, 1, 63, 1.0, (5, 64), softmax_scale_192())
    inp = make_inputs(wl, seed=0)
    kv = inp["kv_len"].numpy()
    assert kv.min() >= 5 and kv.max() <= 64
    out = oracle_rows(inp["q_nope"], inp["q_pe"], inp["k_nope"], inp["k_pe_shared"], inp["v"],
                      inp["kv_len"], inp["past_len"], inp["softmax_scale"])
    assert np.isfinite(out).all()
