"""Pins of the oracle's 2D padding mask (key_mask [B, Tk], 0 = key hidden).

The page "Kimi K2 · Causal mask" (section Construct causal mask) passes the model's 2D
attention_mask into the builder of the 4D mask, which merges it with the causal mask; a
hidden key then carries the dtype minimum like a causally hidden one.  Pins:
  - an all-ones mask changes nothing;
  - torch's float64 scaled_dot_product_attention with the same additive minimum agrees
    (left padding, random holes, ragged kv_len, past_len > 0);
  - for a decode row (causality vacuous), hiding keys equals deleting them;
  - a row with every key hidden has uniform weights over all Tk keys (each score is
    absorbed into the minimum), so its output is the plain mean of the Tk value rows;
  - a pure-Python brute-force loop on tiny shapes.
"""
import math

import numpy as np
import pytest
import torch

from oracle import oracle_rows
from mla_causal_attention_gb300.inputs import make_inputs
from mla_causal_attention_gb300.workloads import Workload, softmax_scale_192

MIN_BF16 = float(torch.finfo(torch.bfloat16).min)


def _inp(B, H, Tq, past, kv=None, seed=0):
    return make_inputs(Workload("t", B, H, Tq, past, 1.0, kv, softmax_scale_192()), seed=seed)


def _rows(inp, mask, rows=None):
    return oracle_rows(inp["q_nope"], inp["q_pe"], inp["k_nope"], inp["k_pe_shared"], inp["v"],
                       inp["kv_len"], inp["past_len"], inp["softmax_scale"], rows=rows,
                       key_mask=mask)


def _visible(inp, mask):
    B, H, Tq = inp["q_nope"].shape[:3]
    Tk = inp["k_nope"].shape[2]
    i = np.arange(Tq)[:, None]
    j = np.arange(Tk)[None, :]
    kvl = np.full(B, Tk) if inp["kv_len"] is None else inp["kv_len"].numpy()
    vis = np.zeros((B, Tq, Tk), dtype=bool)
    for b in range(B):
        vis[b] = (j <= i + inp["past_len"]) & (j < kvl[b]) & (mask[b][None, :] != 0)
    return vis


def _masks(B, Tk, seed):
    rng = np.random.default_rng(seed)
    left = np.ones((B, Tk), dtype=np.uint8)
    for b in range(B):
        left[b, : rng.integers(0, Tk // 2 + 1)] = 0          # left padding
    holes = (rng.random((B, Tk)) > 0.3).astype(np.uint8)      # arbitrary zeros
    return left, holes


def test_all_ones_mask_is_no_mask():
    inp = _inp(2, 3, 5, 4, kv=(3, 9), seed=3)
    ones = np.ones((2, 9), dtype=np.uint8)
    np.testing.assert_array_equal(_rows(inp, ones), _rows(inp, None))


@pytest.mark.parametrize("B,H,Tq,past,kv", [(2, 2, 6, 0, None), (3, 2, 4, 5, (3, 9)),
                                            (2, 3, 1, 11, (4, 12))])
def test_sdpa_float64_with_additive_minimum(B, H, Tq, past, kv):
    inp = _inp(B, H, Tq, past, kv, seed=4)
    Tk = past + Tq
    for mask in _masks(B, Tk, seed=B * 10 + Tq):
        vis = torch.from_numpy(_visible(inp, mask))               # [B, Tq, Tk]
        add = torch.where(vis, 0.0, MIN_BF16).to(torch.float64)[:, None]
        q = torch.cat([inp["q_nope"], inp["q_pe"]], -1).double()
        k = torch.cat([inp["k_nope"], inp["k_pe_shared"][:, None].expand(B, H, Tk, 64)],
                      -1).double()
        v = inp["v"].double()
        scale = float(np.float32(inp["softmax_scale"]))
        ref = torch.nn.functional.scaled_dot_product_attention(q, k, v, attn_mask=add,
                                                               scale=scale)
        np.testing.assert_allclose(_rows(inp, mask), ref.reshape(-1, 128).numpy(), rtol=0,
                                   atol=1e-12)


def test_hiding_a_decode_key_equals_deleting_it():
    B, H, Tk = 2, 2, 13
    inp = _inp(B, H, 1, Tk - 1, None, seed=5)
    mask = np.ones((B, Tk), dtype=np.uint8)
    keep = [0, 2, 3, 7, 8, 12]
    mask[:, [j for j in range(Tk) if j not in keep]] = 0
    got = _rows(inp, mask)
    small = dict(inp)
    for name in ("k_nope", "v"):
        small[name] = inp[name][:, :, keep].contiguous()
    small["k_pe_shared"] = inp["k_pe_shared"][:, keep].contiguous()
    small["past_len"] = len(keep) - 1
    small["kv_len"] = None
    want = _rows(small, None)
    np.testing.assert_allclose(got, want, rtol=0, atol=1e-14)


def test_row_with_every_key_hidden_is_the_mean_of_all_values():
    B, H, Tq, past = 2, 2, 6, 3
    inp = _inp(B, H, Tq, past, None, seed=6)
    Tk = past + Tq
    mask = np.ones((B, Tk), dtype=np.uint8)
    mask[0, :6] = 0   # sequence 0: queries 0..2 (positions 3..5) see no visible key
    got = _rows(inp, mask).reshape(B, H, Tq, 128)
    v = inp["v"].double().numpy()
    for h in range(H):
        for i in range(3):
            np.testing.assert_allclose(got[0, h, i], v[0, h].mean(0), rtol=0, atol=1e-13)
    # the next query sees key 6 only
    np.testing.assert_allclose(got[0, :, 3], v[0, :, 6], rtol=0, atol=1e-13)
    # sequence 1 is unmasked
    np.testing.assert_array_equal(got[1], _rows(inp, None).reshape(B, H, Tq, 128)[1])


def test_brute_force_loop():
    B, H, Tq, past = 2, 2, 3, 2
    inp = _inp(B, H, Tq, past, (2, 5), seed=7)
    Tk = past + Tq
    mask = np.array([[1, 0, 1, 1, 0], [0, 0, 1, 0, 1]], dtype=np.uint8)
    got = _rows(inp, mask).reshape(B, H, Tq, 128)
    qn, qr = inp["q_nope"].double().numpy(), inp["q_pe"].double().numpy()
    kn, kr = inp["k_nope"].double().numpy(), inp["k_pe_shared"].double().numpy()
    v = inp["v"].double().numpy()
    kvl = inp["kv_len"].numpy()
    scale = float(np.float32(inp["softmax_scale"]))
    for b in range(B):
        for h in range(H):
            for i in range(Tq):
                s = []
                for j in range(Tk):
                    dot = math.fsum(qn[b, h, i, d] * kn[b, h, j, d] for d in range(128))
                    dot += math.fsum(qr[b, h, i, d] * kr[b, j, d] for d in range(64))
                    vis = j <= i + past and j < kvl[b] and mask[b, j]
                    s.append(dot * scale + (0.0 if vis else MIN_BF16))
                mx = max(s)
                e = [math.exp(x - mx) for x in s]
                tot = math.fsum(e)
                want = [math.fsum(e[j] / tot * v[b, h, j, d] for j in range(Tk))
                        for d in range(128)]
                np.testing.assert_allclose(got[b, h, i], want, rtol=0, atol=1e-12)
