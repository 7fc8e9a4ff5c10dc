"""Decode path (Tq == 1, split-KV + combine) against the fp64 oracle."""
import pytest
import torch

from mla_causal_attention_gb300.binding import PATH_DECODE
from mla_causal_attention_gb300.inputs import make_inputs
from mla_causal_attention_gb300.workloads import WORKLOADS, Workload, softmax_scale_192
from gpu_helpers import assert_close, gpu_rows, oracle_for, run_gpu, to_device

pytestmark = pytest.mark.gpu


def wl(B, H, past, kv=None, vs=1.0):
    return Workload("t", B, H, 1, past, vs, kv, softmax_scale_192())


@pytest.mark.parametrize("chunk", [0, 64, 128, 1024])
def test_decode_p1000_full(chunk):
    inp = make_inputs(WORKLOADS["decode_p1000"], seed=0)
    out = run_gpu(to_device(inp), path=PATH_DECODE, decode_chunk=chunk)
    assert_close(gpu_rows(out), oracle_for(inp), f"decode_p1000 chunk={chunk}")


@pytest.mark.parametrize("B,H,past,kv,chunk", [
    (3, 5, 76, (1, 77), 0),       # head count not a multiple of the head group
    (2, 8, 299, (100, 300), 64),  # several splits, ragged last split
    (4, 3, 0, None, 0),           # a single key
    (2, 64, 2047, (1, 2048), 256),
    (5, 4, 33, (30, 34), 64),
    (300, 8, 63, (1, 64), 0),     # 600 head groups: the large configuration, one split
])
def test_decode_small_full(B, H, past, kv, chunk):
    inp = make_inputs(wl(B, H, past, kv), seed=1)
    out = run_gpu(to_device(inp), decode_chunk=chunk)
    assert_close(gpu_rows(out), oracle_for(inp), f"decode B{B} H{H} Tk{past + 1}")


def test_decode_ragged_small_batch():
    w = WORKLOADS["decode_ragged"].with_(B=6, past_len=1499, kv_len_range=(200, 1500))
    inp = make_inputs(w, seed=0)
    out = run_gpu(to_device(inp))
    assert_close(gpu_rows(out), oracle_for(inp), "decode_ragged B6")


def test_decode_ragged_full_size_every_row():
    """Configuration 3 at its full size (64 x 64 heads, kv_len in [512, 8192]): every output
    row against the oracle."""
    w = WORKLOADS["decode_ragged"]
    inp = make_inputs(w, seed=0)
    out = run_gpu(to_device(inp))
    assert_close(gpu_rows(out), oracle_for(inp), "decode_ragged every row")


def test_decode_calls_with_changing_plans_share_a_workspace():
    """Calls of different shapes and split plans follow one another on one workspace: each
    call overwrites every partial it reads."""
    from mla_causal_attention_gb300 import binding
    ws = binding.Workspace()
    cases = [wl(8, 64, 2047, (100, 2048)), wl(1, 64, 1000), wl(3, 5, 299, (1, 300)),
             wl(8, 64, 2047, (100, 2048))]
    for k, w in enumerate(cases):
        inp = make_inputs(w, seed=40 + k)
        out = run_gpu(to_device(inp), workspace=ws)
        assert binding.mla_attn_get_status(ws) == 0
        assert_close(gpu_rows(out), oracle_for(inp), f"decode sequence call {k}")


def test_decode_long_context_every_row():
    """One sequence with 131072 cached keys (4.3 GB of keys and values): the scheduler's
    widest splits, every output row against the oracle."""
    inp = make_inputs(wl(1, 64, 131071), seed=6)
    out = run_gpu(to_device(inp))
    assert_close(gpu_rows(out), oracle_for(inp), "decode Tk=131072")


def test_decode_many_sequences_every_row():
    """128 sequences x 64 heads with short ragged caches: 2048 head groups (13 waves of the
    large configuration), one split each."""
    inp = make_inputs(wl(128, 64, 47, (1, 48)), seed=7)
    out = run_gpu(to_device(inp))
    assert_close(gpu_rows(out), oracle_for(inp), "decode B=128 Tk<=48")


def test_decode_single_key_is_exact():
    inp = make_inputs(wl(3, 8, 40, (1, 1)), seed=2)
    inp["kv_len"][:] = 1
    out = run_gpu(to_device(inp))
    assert torch.equal(out.cpu()[:, :, 0, :], inp["v"][:, :, 0, :])


def test_decode_hidden_keys_do_not_matter():
    inp = make_inputs(wl(3, 8, 299, (50, 250)), seed=3)
    base = run_gpu(to_device(inp), decode_chunk=64).cpu()
    for b in range(3):
        k = int(inp["kv_len"][b])
        inp["k_nope"][b, :, k:] = 1e30
        inp["k_pe_shared"][b, k:] = -1e30
        inp["v"][b, :, k:] = 1e30
    again = run_gpu(to_device(inp), decode_chunk=64).cpu()
    assert torch.equal(base, again)


def test_decode_equal_scores_give_mean():
    inp = make_inputs(wl(2, 4, 599, (300, 600)), seed=4)
    inp["q_nope"].zero_()
    inp["q_pe"].zero_()
    out = run_gpu(to_device(inp), decode_chunk=128).float().cpu()
    for b in range(2):
        k = int(inp["kv_len"][b])
        want = inp["v"][b, :, :k].double().mean(dim=1)
        assert (out[b, :, 0].double() - want).abs().max() < 8e-3
