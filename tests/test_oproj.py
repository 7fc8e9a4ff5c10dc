"""Output projection (mla_oproj_fwd) against the fp64 oracle.

o_proj maps the 64 heads' concatenated 128-wide outputs to hidden_size (the MLA init excerpt
on "Kimi K2 · Similarities", section "Scale scores"; 7168, no bias, in the config.json excerpt
on "Kimi K2 · Logits").  The kernel reads the attention output in place ([B,H,T,128]).
Cases: ragged row tiles (T not a multiple of 128), N not a multiple of the column tile,
decode rows (T = 1, more and fewer than 128 sequences), each column-tile width (48, 64,
256), the model's widths sampled, and the attention output of the library itself fed
through.
"""
import numpy as np
import pytest
import torch

from mla_causal_attention_gb300 import binding
from gpu_helpers import assert_close
from oracle import oracle_oproj_rows

pytestmark = pytest.mark.gpu


def _inputs(B, H, T, N, seed):
    g = torch.Generator().manual_seed(seed)
    attn = torch.randn((B, H, T, 128), generator=g).to(torch.bfloat16)
    w = (torch.randn((N, H * 128), generator=g) * (H * 128) ** -0.5).to(torch.bfloat16)
    return attn, w


def _check(B, H, T, N, seed, rows=None, label=""):
    attn, w = _inputs(B, H, T, N, seed)
    y = binding.mla_oproj_fwd(attn.cuda(), w.cuda())
    torch.cuda.synchronize()
    got = y.float().cpu().numpy().reshape(B * T, N).astype(np.float64)
    if rows is not None:
        got = got[rows]
    want = oracle_oproj_rows(attn, w, rows=rows)
    assert_close(got, want, label or f"oproj B{B} H{H} T{T} N{N}")
    return got


@pytest.mark.parametrize("B,H,T,N", [
    (1, 2, 5, 64),        # one ragged row tile, narrow columns
    (2, 3, 130, 96),      # row tiles past T, N below one column tile
    (2, 4, 256, 544),     # two full row tiles, N = 2 x 256 + 32
    (3, 64, 16, 288),     # the tiny-prefill shape's 16 rows
    (5, 8, 1, 64),        # decode rows: 5 sequences
    (200, 4, 1, 320),     # decode rows over two 128-sequence tiles
    (1, 1, 1, 32),        # the smallest: one head (two k-blocks), 32 outputs
    (3, 1, 200, 32),      # one head, ragged row tiles, N below every column tile
    (64, 8, 1, 4096),     # 64 decode rows, every one checked; ragged last column tile
    (33, 16, 1, 7168),    # an odd decode batch at the model width, every row
    (65, 4, 1, 96),       # 65 decode rows
])
def test_oproj_matches_oracle(B, H, T, N):
    _check(B, H, T, N, seed=B * 7 + T)


def test_oproj_wide_tiles_ragged_rows_every_row():
    """Enough row tiles for the 256-column tile path, T not a multiple of 128."""
    _check(2, 4, 1000, 4096, seed=5, label="oproj 256-column tiles")


def test_oproj_kimi_widths_decode_every_row():
    """The bench's decode shape: 64 rows of 64 heads x 128 projected to 7168, every row."""
    _check(64, 64, 1, 7168, seed=3, label="oproj decode widths")


def test_oproj_two_decode_row_tiles_model_width_every_row():
    """130 sequences: two row tiles at the 7168 width take the 64-column tile path."""
    _check(130, 16, 1, 7168, seed=6, label="oproj 64-column tiles")


def test_oproj_kimi_widths_prefill_every_row():
    """The bench's prefill shape: 4096 rows of 64 heads x 128 projected to 7168, every row."""
    _check(1, 64, 4096, 7168, seed=4, label="oproj prefill widths")


def test_oproj_of_the_attention_output():
    """The attention core's own output projected: the two calls chain with no reshape."""
    from mla_causal_attention_gb300.inputs import make_inputs
    from mla_causal_attention_gb300.workloads import Workload, softmax_scale_192
    inp = make_inputs(Workload("t", 2, 8, 40, 0, 1.0, None, softmax_scale_192()), seed=11)
    d = {k: inp[k].cuda() for k in ("q_nope", "q_pe", "k_nope", "k_pe_shared", "v")}
    attn = binding.mla_attn_fwd(d["q_nope"], d["q_pe"], d["k_nope"], d["k_pe_shared"], d["v"],
                                None, inp["past_len"], inp["softmax_scale"])
    g = torch.Generator().manual_seed(12)
    w = (torch.randn((256, 8 * 128), generator=g) * (8 * 128) ** -0.5).to(torch.bfloat16)
    y = binding.mla_oproj_fwd(attn, w.cuda())
    torch.cuda.synchronize()
    got = y.float().cpu().numpy().reshape(-1, 256).astype(np.float64)
    want = oracle_oproj_rows(attn.cpu(), w)  # projection of exactly what the kernel produced
    assert_close(got, want, "oproj of attention output")
