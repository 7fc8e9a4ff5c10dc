"""Pins of the oracle's output projection (o_proj: nn.Linear from num_heads x v_head_dim to
hidden_size, the MLA init excerpt on "Kimi K2 · Similarities", section "Scale scores"; no
bias, attention_bias false in the config.json excerpt on "Kimi K2 · Logits").

The oracle is pinned against things other than itself: numpy's float64 matrix product on
the head-concatenated rows (a library routine), selection weights whose outputs are single
input features (exact), exact scaling, and the row subset.  Reading of the layout: input
feature k = h * 128 + d (heads concatenated in head order).
"""
import numpy as np
import pytest
import torch

from oracle import oracle_oproj_rows, round_bf16

pytestmark = pytest.mark.filterwarnings("ignore")


def _bf16(shape, gen, scale=1.0):
    return (torch.randn(shape, generator=gen) * scale).to(torch.bfloat16)


def _as_f64(t):
    return t.float().double().numpy()


def _concat_rows(attn):
    """[B,H,T,128] -> [B*T, H*128], row (b, i), feature h*128 + d."""
    a = _as_f64(attn)
    B, H, T, D = a.shape
    return a.transpose(0, 2, 1, 3).reshape(B * T, H * D)


def test_matches_numpy_matmul_on_concatenated_heads():
    g = torch.Generator().manual_seed(5)
    B, H, T, N = 2, 3, 5, 24
    attn = _bf16((B, H, T, 128), g)
    w = _bf16((N, H * 128), g, 128 ** -0.5)
    got = oracle_oproj_rows(attn, w, threads=2)
    want = _concat_rows(attn) @ _as_f64(w).T
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12)


def test_selection_weights_return_single_features_exactly():
    """W[n, k_n] = 1, all else 0: y[:, n] = x[:, k_n].  Features are picked from every head
    and both halves of the 128 columns, so the head order and the column index are pinned."""
    g = torch.Generator().manual_seed(6)
    B, H, T = 2, 4, 3
    attn = _bf16((B, H, T, 128), g)
    rng = np.random.default_rng(0)
    picks = [h * 128 + d for h in range(H) for d in (0, 1, 63, 64, 127)]
    picks += rng.integers(0, H * 128, 11).tolist()
    N = len(picks)
    w = torch.zeros((N, H * 128), dtype=torch.bfloat16)
    for n, k in enumerate(picks):
        w[n, k] = 1.0
    got = oracle_oproj_rows(attn, w, threads=3)
    x = _concat_rows(attn)
    assert np.array_equal(got, x[:, picks])


def test_exact_scaling_and_zero_weight():
    g = torch.Generator().manual_seed(7)
    B, H, T, N = 1, 2, 4, 16
    attn = _bf16((B, H, T, 128), g)
    w = _bf16((N, H * 128), g, 0.1)
    y1 = oracle_oproj_rows(attn, w)
    y2 = oracle_oproj_rows((attn.float() * 2).to(torch.bfloat16), w)  # exact in bf16
    assert np.array_equal(y2, 2 * y1)
    assert not np.any(oracle_oproj_rows(attn, torch.zeros_like(w)))


def test_row_subset_and_row_order():
    g = torch.Generator().manual_seed(8)
    B, H, T, N = 3, 2, 7, 8
    attn = _bf16((B, H, T, 128), g)
    w = _bf16((N, H * 128), g, 0.1)
    full = oracle_oproj_rows(attn, w)
    rows = [20, 0, 7, 13, 6]
    np.testing.assert_array_equal(oracle_oproj_rows(attn, w, rows=rows), full[rows])
    # row r = b * T + i: a change in (b=1, i=3) moves only that row
    a2 = attn.clone()
    a2[1, :, 3, :] = 0
    diff = np.any(oracle_oproj_rows(a2, w) != full, axis=1)
    assert diff.tolist() == [r == 1 * T + 3 for r in range(B * T)]


def test_kimi_k2_width_row():
    """One row at the model's widths (64 heads x 128 -> 7168) against numpy."""
    g = torch.Generator().manual_seed(9)
    attn = _bf16((1, 64, 2, 128), g)
    w = _bf16((7168, 64 * 128), g, (64 * 128) ** -0.5)
    got = oracle_oproj_rows(attn, w, rows=[1])
    want = _concat_rows(attn)[1] @ _as_f64(w).T
    np.testing.assert_allclose(got[0], want, rtol=1e-10, atol=1e-10)
    assert round_bf16(1.0) == 1.0
