"""Attention with a 2D padding mask on the keys (mla_attn_masked_fwd) against the oracle.

Covers decode and prefill with left padding, arbitrary holes, ragged kv_len and past_len,
rows that see no visible key (their output is the mean of all value rows), and the
all-ones mask, which must reproduce mla_attn_fwd bit for bit.
"""
import numpy as np
import pytest
import torch

from mla_causal_attention_gb300 import binding
from mla_causal_attention_gb300.inputs import make_inputs
from mla_causal_attention_gb300.workloads import WORKLOADS, Workload, softmax_scale_192
from gpu_helpers import assert_close, gpu_rows, run_gpu, to_device
from oracle import oracle_rows

pytestmark = pytest.mark.gpu


def _mask(B, Tk, kind, seed):
    rng = np.random.default_rng(seed)
    m = np.ones((B, Tk), dtype=np.uint8)
    if kind in ("left", "both"):
        for b in range(B):
            m[b, : rng.integers(0, max(1, Tk // 2))] = 0
    if kind in ("holes", "both"):
        m &= (rng.random((B, Tk)) > 0.25).astype(np.uint8)
    if kind == "none_visible":
        m[0] = 0  # sequence 0: no key visible to any row
    return m


def _run(inp, mask):
    d = to_device(inp)
    km = torch.from_numpy(mask).cuda()
    out = binding.mla_attn_masked_fwd(d["q_nope"], d["q_pe"], d["k_nope"], d["k_pe_shared"],
                                      d["v"], d["kv_len"], km, inp["past_len"],
                                      inp["softmax_scale"])
    torch.cuda.synchronize()
    assert binding.mla_attn_get_status(device=out.device) == 0
    return out


def _oracle(inp, mask, rows=None):
    return oracle_rows(inp["q_nope"], inp["q_pe"], inp["k_nope"], inp["k_pe_shared"],
                       inp["v"], inp["kv_len"], inp["past_len"], inp["softmax_scale"],
                       rows=rows, key_mask=mask)


@pytest.mark.parametrize("B,H,Tq,past,kv,kind", [
    (3, 8, 1, 299, None, "left"),          # decode, several splits
    (3, 8, 1, 299, (50, 300), "holes"),    # decode, ragged
    (2, 4, 1, 4000, None, "both"),         # decode, long cache
    (2, 4, 1, 99, None, "none_visible"),   # decode row with no visible key
    (1, 64, 1, 1000, None, "holes"),       # the decode shape at cached length 1000
    (2, 3, 130, 77, None, "left"),         # prefill: left padding hides early query rows
    (2, 3, 130, 77, (100, 207), "both"),   # prefill, ragged + holes
    (2, 2, 300, 0, None, "left"),          # prefill from an empty cache, degenerate rows
    (2, 2, 256, 5, None, "none_visible"),  # prefill sequence with nothing visible
    (1, 4, 513, 1000, None, "holes"),      # prefill with a long cached prefix
])
def test_masked_matches_oracle(B, H, Tq, past, kv, kind):
    inp = make_inputs(Workload("t", B, H, Tq, past, 1.0, kv, softmax_scale_192()), seed=31)
    mask = _mask(B, past + Tq, kind, seed=B * 7 + Tq)
    out = _run(inp, mask)
    assert_close(gpu_rows(out), _oracle(inp, mask), f"mask {kind} B{B} H{H} Tq{Tq} p{past}")


@pytest.mark.parametrize("B,H,Tq,past,kv", [(3, 8, 1, 299, (50, 300)), (2, 3, 130, 77, (100, 207))])
def test_all_ones_mask_equals_unmasked(B, H, Tq, past, kv):
    inp = make_inputs(Workload("t", B, H, Tq, past, 1.0, kv, softmax_scale_192()), seed=32)
    ones = np.ones((B, past + Tq), dtype=np.uint8)
    assert torch.equal(_run(inp, ones).cpu(), run_gpu(to_device(inp)).cpu())


def test_rows_with_no_visible_key_are_value_means():
    B, H, Tq, past = 2, 4, 40, 8
    inp = make_inputs(Workload("t", B, H, Tq, past, 1.0, None, softmax_scale_192()), seed=33)
    mask = np.ones((B, Tk := past + Tq), dtype=np.uint8)
    mask[1, :20] = 0  # sequence 1: rows i with i + 8 < 20 see nothing
    out = _run(inp, mask).float().cpu().numpy()
    mean = inp["v"].double().numpy()[1].mean(1)  # [H, 128]
    for i in range(12):
        np.testing.assert_allclose(out[1, :, i], mean, rtol=0, atol=1e-2)


def test_long_prefill_left_padded_every_row():
    """The long prefill (8 heads) with its first 700 keys hidden: rows 0..699 see no key
    (value means), every row against the oracle."""
    w = WORKLOADS["long_prefill"].with_(H=8)
    inp = make_inputs(w, seed=0)
    mask = np.ones((1, w.Tk), dtype=np.uint8)
    mask[0, :700] = 0
    out = _run(inp, mask)
    assert_close(gpu_rows(out), _oracle(inp, mask), "long_prefill left pad 700, every row")


@pytest.mark.parametrize("B,H,Tq,past,pads", [
    (2, 4, 384, 200, (300, 520)),  # prefill: whole leading key tiles hidden (skipped)
    (1, 4, 640, 0, (385,)),        # prefill from an empty cache: three tiles and one key
    (5, 64, 1, 99, (100, 0, 3, 0, 0)),  # decode, sequence 0 sees nothing; B*H above the SMs
    (20, 16, 16, 40, (56,)),       # prefill, sequence 0 sees nothing; B*H above the SMs
])
def test_left_padding_whole_tiles(B, H, Tq, past, pads):
    """Left padding that covers whole 128-key tiles, and rows with nothing visible in
    batches large enough that one pass over the value rows serves several heads."""
    inp = make_inputs(Workload("t", B, H, Tq, past, 1.0, None, softmax_scale_192()), seed=34)
    mask = np.ones((B, past + Tq), dtype=np.uint8)
    for b, n in enumerate(pads):
        mask[b, :n] = 0
    out = _run(inp, mask)
    assert_close(gpu_rows(out), _oracle(inp, mask), f"left pads {pads} B{B} H{H} Tq{Tq}")
