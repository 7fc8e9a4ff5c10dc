"""Prefill path (tcgen05 / TMEM / TMA kernel) against the fp64 oracle."""
import pytest
import torch

from mla_causal_attention_gb300.binding import PATH_PREFILL
from mla_causal_attention_gb300.inputs import make_inputs
from mla_causal_attention_gb300.workloads import WORKLOADS, Workload, softmax_scale_192
from gpu_helpers import assert_close, gpu_rows, oracle_for, run_gpu, to_device

pytestmark = pytest.mark.gpu


def wl(B, H, Tq, past, kv=None, vs=1.0):
    return Workload("t", B, H, Tq, past, vs, kv, softmax_scale_192())


def test_tiny_prefill_full():
    inp = make_inputs(WORKLOADS["tiny_prefill"], seed=0)
    out = run_gpu(to_device(inp))
    assert_close(gpu_rows(out), oracle_for(inp), "tiny_prefill")


@pytest.mark.parametrize("B,H,Tq,past,kv", [
    (1, 2, 1, 0, None),        # one query through the prefill path
    (1, 2, 2, 0, None),
    (2, 3, 17, 0, None),
    (1, 2, 129, 0, None),      # one row past a tile
    (1, 2, 255, 5, None),
    (1, 2, 256, 0, None),      # exactly one tile pair
    (1, 2, 257, 3, None),      # ragged second pair
    (2, 2, 300, 77, (200, 377)),  # padding inside the causal range, unaligned past_len
    (1, 4, 512, 1000, None),   # many key tiles before the diagonal
    (3, 2, 130, 126, (5, 256)),
    (40, 8, 16, 10, (1, 26)),  # 320 units: every CTA walks several; kv_len ragged in [1, 26]
])
def test_prefill_shapes_full(B, H, Tq, past, kv):
    inp = make_inputs(wl(B, H, Tq, past, kv), seed=5)
    out = run_gpu(to_device(inp), path=PATH_PREFILL)
    assert_close(gpu_rows(out), oracle_for(inp), f"prefill B{B} H{H} Tq{Tq} past{past}")


def test_chunked_prefill_small_full():
    inp = make_inputs(wl(2, 4, 384, 640, (900, 1024)), seed=6)
    out = run_gpu(to_device(inp))
    assert_close(gpu_rows(out), oracle_for(inp), "chunked small")


def test_long_prefill_full_size_every_row():
    """Configuration 4 at its full size: all 64 x 4096 output rows against the oracle."""
    w = WORKLOADS["long_prefill"]
    inp = make_inputs(w, seed=0)
    out = run_gpu(to_device(inp))
    assert_close(gpu_rows(out), oracle_for(inp), "long_prefill every row")


def test_chunked_prefill_full_size_every_row():
    """Configuration 5 at its full size: all 4 x 64 x 2048 output rows against the oracle."""
    w = WORKLOADS["chunked_prefill"]
    inp = make_inputs(w, seed=0)
    out = run_gpu(to_device(inp))
    assert_close(gpu_rows(out), oracle_for(inp), "chunked_prefill every row")


def test_prefill_long_sequence_every_row():
    """8192 new rows on 8192 cached ones (Tk = 16384, 64 key tiles per query tile at the
    end), two heads: every output row against the oracle."""
    inp = make_inputs(wl(1, 2, 8192, 8192), seed=11)
    out = run_gpu(to_device(inp))
    assert_close(gpu_rows(out), oracle_for(inp), "prefill Tq=8192 past=8192")


def test_prefill_many_units_every_row():
    """64 sequences x 64 heads x 300 rows: 8192 work units over the persistent grid, ragged
    kv_len inside the causal range."""
    inp = make_inputs(wl(64, 64, 300, 20, (100, 320)), seed=12)
    out = run_gpu(to_device(inp))
    assert_close(gpu_rows(out), oracle_for(inp), "prefill B64 H64 Tq300")


def test_prefill_first_row_is_exact():
    inp = make_inputs(wl(2, 3, 200, 0), seed=7)
    out = run_gpu(to_device(inp)).cpu()
    assert torch.equal(out[:, :, 0, :], inp["v"][:, :, 0, :])


def test_prefill_hidden_keys_do_not_matter():
    w = wl(2, 2, 300, 100, (250, 400))
    inp = make_inputs(w, seed=8)
    base = run_gpu(to_device(inp)).cpu()
    for b in range(2):
        k = int(inp["kv_len"][b])
        inp["k_nope"][b, :, k:] = 1e30
        inp["k_pe_shared"][b, k:] = -1e30
        inp["v"][b, :, k:] = 1e30
    again = run_gpu(to_device(inp)).cpu()
    assert torch.equal(base, again)
    # causal part: keys after the last query's position never matter for row 0..9
    inp2 = make_inputs(wl(1, 2, 260, 0), seed=9)
    ref = run_gpu(to_device(inp2)).cpu()
    inp2["k_nope"][0, :, 10:] = 1e30
    inp2["v"][0, :, 10:] = -1e30
    inp2["k_pe_shared"][0, 10:] = 1e30
    out = run_gpu(to_device(inp2)).cpu()
    assert torch.equal(out[0, :, :10], ref[0, :, :10])


def test_prefill_equal_scores_give_mean():
    w = wl(1, 2, 300, 40)
    inp = make_inputs(w, seed=10)
    inp["q_nope"].zero_()
    inp["q_pe"].zero_()
    out = run_gpu(to_device(inp)).double().cpu()
    v = inp["v"].double()
    for i in (0, 1, 100, 299):
        want = v[0, :, : i + 41].mean(dim=1)
        assert (out[0, :, i] - want).abs().max() < 8e-3
