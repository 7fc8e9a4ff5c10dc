"""Pins of the oracle's latent-cache rows (the kv_b_proj up-projection, "Kimi K2 ·
Similarities", §Scale scores: kv_lora_rank 512 -> 64 heads x (128 no-rope key + 128 value)).

  - With selection weights (head h's no-rope key = latent dims [8h, 8h + 128), its value =
    dims [256 + 16h, 256 + 16h + 128)) the rows equal the standard attention oracle on
    those explicitly built per-head keys and values: pins which weight rows are keys and
    which are values, the per-head indexing, and that the rotary key still adds in.
  - Doubling the value rows of the weight doubles the output (exact in bf16 and fp64).
  - A query that sees one key returns W_V[h] . c_0 (closed form).
"""
import numpy as np
import pytest
import torch

from oracle import oracle_latent_rows, oracle_rows
from mla_causal_attention_gb300.workloads import softmax_scale_192


def _lat_case(B, H, Tq, past, seed, kv=None):
    g = torch.Generator("cpu").manual_seed(seed)
    Tk = past + Tq
    mk = lambda *s: torch.randn(*s, generator=g).to(torch.bfloat16)  # noqa: E731
    d = dict(q_nope=mk(B, H, Tq, 128), q_pe=mk(B, H, Tq, 64), c_kv=mk(B, Tk, 512),
             k_pe=mk(B, Tk, 64), w_kvb=(torch.randn(H * 256, 512, generator=g) / 22.6)
             .to(torch.bfloat16), kv_len=None, past_len=past)
    if kv is not None:
        d["kv_len"] = torch.randint(kv[0], kv[1] + 1, (B,), generator=g, dtype=torch.int32)
    return d


def _lat(d, rows=None):
    return oracle_latent_rows(d["q_nope"], d["q_pe"], d["c_kv"], d["k_pe"], d["w_kvb"],
                              d["kv_len"], d["past_len"], softmax_scale_192(), rows=rows)


@pytest.mark.parametrize("B,H,Tq,past,kv", [(2, 3, 1, 9, (3, 10)), (1, 2, 5, 4, None)])
def test_selection_weights_reduce_to_standard_attention(B, H, Tq, past, kv):
    d = _lat_case(B, H, Tq, past, seed=1, kv=kv)
    Tk = past + Tq
    w = torch.zeros(H * 256, 512)
    for h in range(H):
        for e in range(128):
            w[h * 256 + e, 8 * h + e] = 1.0
            w[h * 256 + 128 + e, 256 + 16 * h + e] = 1.0
    d["w_kvb"] = w.to(torch.bfloat16)
    c = d["c_kv"]
    k_nope = torch.stack([c[:, :, 8 * h: 8 * h + 128] for h in range(H)], 1).contiguous()
    v = torch.stack([c[:, :, 256 + 16 * h: 256 + 16 * h + 128] for h in range(H)], 1).contiguous()
    want = oracle_rows(d["q_nope"], d["q_pe"], k_nope, d["k_pe"], v, d["kv_len"], past,
                       softmax_scale_192())
    np.testing.assert_allclose(_lat(d), want, rtol=0, atol=1e-12)
    assert Tk == k_nope.shape[2]


def test_doubling_value_weights_doubles_output():
    d = _lat_case(2, 2, 1, 6, seed=2)
    a = _lat(d)
    w = d["w_kvb"].clone().view(2, 256, 512)
    w[:, 128:] *= 2
    d["w_kvb"] = w.view(512, 512)
    np.testing.assert_allclose(_lat(d), 2 * a, rtol=0, atol=1e-12)


def test_single_visible_key_is_projected_latent():
    d = _lat_case(1, 3, 3, 0, seed=3)  # query 0 sees key 0 only
    out = _lat(d, rows=[h * 3 for h in range(3)])
    w = d["w_kvb"].double().numpy().reshape(3, 256, 512)
    c0 = d["c_kv"].double().numpy()[0, 0]
    for h in range(3):
        np.testing.assert_allclose(out[h], w[h, 128:] @ c0, rtol=0, atol=1e-12)


def test_two_keys_weighted_by_the_rotary_part_alone():
    """With the no-rope key rows of the weight zero, the scores come from the shared rotary
    key only: a query that sees keys 0 and 1 returns w0 v0 + w1 v1 with
    w0 = 1 / (1 + exp(scale (q_pe . k_pe_1 - q_pe . k_pe_0))) and v_j = W_V[h] . c_j."""
    d = _lat_case(1, 2, 1, 1, seed=4)  # Tk = 2, the query (position 1) sees both keys
    w = d["w_kvb"].clone().view(2, 256, 512)
    w[:, :128] = 0
    d["w_kvb"] = w.view(512, 512)
    out = _lat(d)
    sc = float(np.float32(softmax_scale_192()))
    qp = d["q_pe"].double().numpy()[0, :, 0]        # [H, 64]
    kp = d["k_pe"].double().numpy()[0]               # [2, 64]
    c = d["c_kv"].double().numpy()[0]                # [2, 512]
    wv = d["w_kvb"].double().numpy().reshape(2, 256, 512)[:, 128:]
    for h in range(2):
        s0, s1 = sc * qp[h] @ kp[0], sc * qp[h] @ kp[1]
        w0 = 1.0 / (1.0 + np.exp(s1 - s0))
        want = w0 * (wv[h] @ c[0]) + (1 - w0) * (wv[h] @ c[1])
        np.testing.assert_allclose(out[h], want, rtol=0, atol=1e-12)
