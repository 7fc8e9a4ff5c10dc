"""Rotary step + cache append + attention (mla_attn_rope_append_fwd) against the fp64 oracle.

The query's and the new keys' rotary parts arrive unrotated and are rotated at position
past_len + t with YaRN frequencies (the rotary calls of the attention excerpt on "Kimi K2 ·
Similarities", the rope_scaling block of the config.json excerpt on "Kimi K2 · Logits").
Checked: the cos/sin table, the output against oracle_rows_rope, the cache contents (new
no-rope key and value rows copied, new rotary key rows rotated, nothing else touched), and
that decoding token by token builds the same cache as one prefill.
"""
import numpy as np
import pytest
import torch

from mla_causal_attention_gb300 import binding
from mla_causal_attention_gb300.inputs import make_inputs
from mla_causal_attention_gb300.workloads import WORKLOADS, Workload, softmax_scale_192
from gpu_helpers import assert_close, errors, gpu_rows
from oracle import oracle_rows_rope, rotate, yarn

pytestmark = pytest.mark.gpu
POISON = 3.0  # finite filler for cache rows beyond the appended ones
PAGE = dict(theta=50000.0, factor=32.0, orig_max_pos=4096, beta_fast=1.0, beta_slow=1.0,
            mscale=1.0, mscale_all_dim=1.0)
RATIO = dict(theta=50000.0, factor=32.0, orig_max_pos=4096, beta_fast=1.0, beta_slow=1.0,
             mscale=1.0, mscale_all_dim=0.707)  # mscale ratio != 1


def _cfg(c):
    return binding.RopeConfig(c["theta"], c["factor"], c["orig_max_pos"], c["beta_fast"],
                              c["beta_slow"], c["mscale"], c["mscale_all_dim"])


def _case(B, H, Tq, past, T_cap, kv=None, seed=0, vs=1.0):
    """Inputs whose k_pe_shared rows < past are the (already rotated) cached rows and rows
    >= past the unrotated new ones; caches on the device hold the prefix and POISON."""
    inp = make_inputs(Workload("t", B, H, Tq, past, vs, kv, softmax_scale_192()), seed=seed)
    Tk = past + Tq
    cache = {}
    for name, shape in (("k_nope", (B, H, T_cap, 128)), ("v", (B, H, T_cap, 128)),
                        ("k_pe_shared", (B, T_cap, 64))):
        c = torch.full(shape, POISON, dtype=torch.bfloat16)
        if name == "k_pe_shared":
            c[:, :past] = inp[name][:, :past]
        else:
            c[:, :, :past] = inp[name][:, :, :past]
        cache[name] = c.cuda()
    new = {"k_nope": inp["k_nope"][:, :, past:Tk].contiguous().cuda(),
           "v": inp["v"][:, :, past:Tk].contiguous().cuda(),
           "k_pe_shared": inp["k_pe_shared"][:, past:Tk].contiguous().cuda()}
    return inp, cache, new


def _run(inp, cache, new, table, kv_len=True):
    """kv_len=False passes no kv_len (every sequence attends to all its keys)."""
    kv = inp["kv_len"].cuda() if kv_len and inp["kv_len"] is not None else None
    out = binding.mla_attn_rope_append_fwd(
        inp["q_nope"].cuda(), inp["q_pe"].cuda(), new["k_nope"], new["k_pe_shared"], new["v"],
        cache["k_nope"], cache["k_pe_shared"], cache["v"], kv, inp["past_len"],
        inp["softmax_scale"], table)
    torch.cuda.synchronize()
    return out


def _oracle(inp, c, rows=None):
    f, r = yarn(**c)
    return oracle_rows_rope(inp["q_nope"], inp["q_pe"], inp["k_nope"], inp["k_pe_shared"],
                            inp["v"], inp["kv_len"], inp["past_len"], inp["softmax_scale"], f,
                            r, rows=rows)


def _check_cache(inp, cache, c, T_cap):
    past = inp["past_len"]
    Tk = inp["k_nope"].shape[2]
    for name in ("k_nope", "v"):
        got = cache[name].cpu()
        assert torch.equal(got[:, :, :Tk], inp[name]), name  # prefix kept, new rows copied
        assert bool((got[:, :, Tk:] == POISON).all()), name
    got = cache["k_pe_shared"].cpu()
    assert torch.equal(got[:, :past], inp["k_pe_shared"][:, :past])
    assert bool((got[:, Tk:] == POISON).all())
    # new rotary key rows: the oracle's rotation at their positions, rounded to bf16 by the
    # kernel (float arithmetic): within one bf16 ulp of the exact value
    f, r = yarn(**c)
    pos = np.arange(past, Tk)[None, :]
    want = rotate(inp["k_pe_shared"][:, past:Tk], pos, f, r)
    g = got[:, past:Tk].double().numpy()
    assert (np.abs(g - want) <= np.abs(want) * 2.0 ** -7 + 1e-6).all()


def test_table_matches_oracle_angles():
    for c in (PAGE, RATIO):
        max_pos = 163840
        table = binding.mla_rope_table(max_pos, _cfg(c))
        torch.cuda.synchronize()
        f, r = yarn(**c)
        pos = np.array([0, 1, 2, 4095, 4096, 65535, 131071, 163839])
        want_c = np.cos(pos[:, None] * f[None, :]) * r
        want_s = np.sin(pos[:, None] * f[None, :]) * r
        got = table[torch.from_numpy(pos).cuda()].double().cpu().numpy()
        np.testing.assert_allclose(got[:, :32], want_c, rtol=0, atol=1.5e-7)
        np.testing.assert_allclose(got[:, 32:], want_s, rtol=0, atol=1.5e-7)


@pytest.mark.parametrize("B,H,Tq,past,T_cap,kv,c", [
    (3, 8, 1, 299, 320, None, PAGE),            # decode, several splits, fused append
    (1, 64, 1, 1000, 1024, None, PAGE),         # the decode shape at cached length 1000
    (3, 4, 1, 99, 128, (50, 100), PAGE),        # ragged: the new row hidden, still written
    (2, 3, 130, 77, 300, None, PAGE),           # prefill: rope pre-pass, then attention
    (2, 2, 256, 0, 256, None, RATIO),           # empty cache, full capacity, ratio != 1
    (1, 2, 3, 100000, 100008, None, PAGE),      # far positions (angles ~ 1e5 rad), prefill
    (2, 4, 1, 120000, 120001, None, RATIO),     # far positions, decode
])
def test_rope_append_matches_oracle_and_writes_cache(B, H, Tq, past, T_cap, kv, c):
    inp, cache, new = _case(B, H, Tq, past, T_cap, kv, seed=41)
    table = binding.mla_rope_table(T_cap, _cfg(c))
    out = _run(inp, cache, new, table)
    assert_close(gpu_rows(out), _oracle(inp, c), f"rope B{B} H{H} Tq{Tq} past{past}")
    _check_cache(inp, cache, c, T_cap)


@pytest.mark.parametrize("B,H,Tq,past,T_cap,c", [
    (2, 3, 130, 0, 300, RATIO),    # empty cache, ratio != 1
    (1, 4, 200, 256, 600, PAGE),   # cached tiles, then rotated new rows
    (2, 2, 129, 128, 257, PAGE),   # capacity exactly Tk
])
def test_rope_append_fused_prefill(B, H, Tq, past, T_cap, c):
    """Prefill on a prefix of whole key tiles without kv_len: the rotary pass only rotates
    (queries, and new rotary keys into the workspace); the attention kernel reads the new
    rows and writes all three into the caches."""
    inp, cache, new = _case(B, H, Tq, past, T_cap, None, seed=43)
    table = binding.mla_rope_table(T_cap, _cfg(c))
    out = _run(inp, cache, new, table, kv_len=False)
    assert_close(gpu_rows(out), _oracle(inp, c), f"fused rope B{B} H{H} Tq{Tq} past{past}")
    _check_cache(inp, cache, c, T_cap)


def test_decode_steps_build_the_same_cache_as_one_prefill():
    B, H, N, T_cap = 2, 4, 40, 64
    inp, cache_p, new = _case(B, H, N, 0, T_cap, None, seed=42)
    table = binding.mla_rope_table(T_cap)
    out_p = _run(inp, cache_p, new, table)
    _, cache_d, _ = _case(B, H, N, 0, T_cap, None, seed=42)
    for t in range(N):
        step = {k: inp[k] for k in ("softmax_scale",)}
        step.update(q_nope=inp["q_nope"][:, :, t:t + 1].contiguous(),
                    q_pe=inp["q_pe"][:, :, t:t + 1].contiguous(), kv_len=None, past_len=t)
        one = {"k_nope": new["k_nope"][:, :, t:t + 1].contiguous(),
               "v": new["v"][:, :, t:t + 1].contiguous(),
               "k_pe_shared": new["k_pe_shared"][:, t:t + 1].contiguous()}
        out_t = _run(step, cache_d, one, table)
        mx, _ = errors(gpu_rows(out_t), gpu_rows(out_p[:, :, t:t + 1]).astype(np.float64))
        assert mx <= 2e-2, (t, mx)
    for k in cache_p:
        assert torch.equal(cache_p[k], cache_d[k]), k


def test_decode_p1000_shape_with_rope():
    w = WORKLOADS["decode_p1000"]
    inp, cache, new = _case(w.B, w.H, 1, w.past_len, 1024, None, seed=0)
    table = binding.mla_rope_table(131072)
    out = _run(inp, cache, new, table)
    assert_close(gpu_rows(out), _oracle(inp, PAGE), "decode_p1000 rope")


def test_long_prefill_with_rope_every_row():
    """The bench's rotary + append prefill (64 heads x 4096 new rows, empty cache): the fused
    call (no kv_len) against the oracle on every row; the copy-first call (with kv_len)
    gives the same bits and the same caches."""
    w = WORKLOADS["long_prefill"]
    inp, cache, new = _case(w.B, w.H, w.Tq, 0, w.Tq, None, seed=0, vs=w.value_scale)
    table = binding.mla_rope_table(w.Tq)
    fused = _run(inp, cache, new, table, kv_len=False)
    assert_close(gpu_rows(fused), _oracle(inp, PAGE), "long_prefill rope fused, every row")
    _check_cache(inp, cache, PAGE, w.Tq)
    _, cache2, _ = _case(w.B, w.H, w.Tq, 0, w.Tq, None, seed=0, vs=w.value_scale)
    copied = _run(inp, cache2, new, table)
    assert torch.equal(fused, copied)
    for k in cache:
        assert torch.equal(cache[k], cache2[k]), k


def test_ragged_decode_with_rope_sampled():
    w = WORKLOADS["decode_ragged"].with_(B=8)
    inp, cache, new = _case(w.B, w.H, 1, w.past_len, w.Tk, w.kv_len_range, seed=0)
    table = binding.mla_rope_table(w.Tk)
    out = _run(inp, cache, new, table)
    rows = [b * w.H + h for b in range(w.B) for h in (0, 17, 63)]
    assert_close(gpu_rows(out, rows), _oracle(inp, PAGE, rows), "decode_ragged B8 rope")
