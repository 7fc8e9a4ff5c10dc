"""Cache append + attention (mla_attn_append_fwd) against the fp64 oracle.

The new key/value rows must land at rows [past_len, past_len + Tq) of the caches (the cache
update of the attention excerpt: new rows after the cached prefix), every other cache row
must be left untouched, and the output must equal attention over the concatenated keys.
"""
import pytest
import torch

from mla_causal_attention_gb300 import binding
from mla_causal_attention_gb300.inputs import make_inputs
from mla_causal_attention_gb300.workloads import Workload, softmax_scale_192
from gpu_helpers import assert_close, gpu_rows, oracle_for, run_gpu, to_device

pytestmark = pytest.mark.gpu
POISON = 3.0  # finite filler for cache rows beyond the appended ones


def _case(B, H, Tq, past, T_cap, kv=None, seed=0):
    wl = Workload("t", B, H, Tq, past, 1.0, kv, softmax_scale_192())
    inp = make_inputs(wl, seed=seed)
    Tk = past + Tq
    dev = "cuda"
    cache = {}
    for name, shape in (("k_nope", (B, H, T_cap, 128)), ("v", (B, H, T_cap, 128)),
                        ("k_pe_shared", (B, T_cap, 64))):
        c = torch.full(shape, POISON, dtype=torch.bfloat16)
        if name == "k_pe_shared":
            c[:, :past] = inp[name][:, :past]
        else:
            c[:, :, :past] = inp[name][:, :, :past]
        cache[name] = c.to(dev)
    new = {"k_nope": inp["k_nope"][:, :, past:Tk].contiguous().to(dev),
           "v": inp["v"][:, :, past:Tk].contiguous().to(dev),
           "k_pe_shared": inp["k_pe_shared"][:, past:Tk].contiguous().to(dev)}
    return wl, inp, cache, new


def _check_cache(inp, cache, past, Tq, T_cap):
    Tk = past + Tq
    for name in ("k_nope", "v"):
        c = cache[name].cpu()
        assert torch.equal(c[:, :, :Tk], inp[name]), name
        assert bool((c[:, :, Tk:] == POISON).all()), name
    c = cache["k_pe_shared"].cpu()
    assert torch.equal(c[:, :Tk], inp["k_pe_shared"])
    assert bool((c[:, Tk:] == POISON).all())


@pytest.mark.parametrize("B,H,Tq,past,T_cap,kv", [
    (3, 8, 1, 299, 320, None),             # decode, several splits, fused append
    (1, 64, 1, 1000, 1024, None),          # the decode shape at cached length 1000
    (3, 4, 1, 99, 128, (50, 100)),         # ragged: the new row may be hidden, still written
    (2, 3, 130, 77, 300, None),            # prefill: copy kernel, then attention
    (2, 2, 256, 0, 256, None),             # prefill into an empty cache, full capacity
])
def test_append_matches_oracle_and_writes_cache(B, H, Tq, past, T_cap, kv):
    wl, inp, cache, new = _case(B, H, Tq, past, T_cap, kv, seed=21)
    d = to_device(inp)
    out = binding.mla_attn_append_fwd(d["q_nope"], d["q_pe"], new["k_nope"],
                                      new["k_pe_shared"], new["v"], cache["k_nope"],
                                      cache["k_pe_shared"], cache["v"], d["kv_len"], past,
                                      inp["softmax_scale"])
    torch.cuda.synchronize()
    assert_close(gpu_rows(out), oracle_for(inp), f"append B{B} H{H} Tq{Tq} past{past}")
    _check_cache(inp, cache, past, Tq, T_cap)


@pytest.mark.parametrize("B,H,Tq,past,T_cap", [
    (2, 3, 130, 0, 300),      # empty cache: every key tile comes from the new rows
    (2, 2, 300, 256, 700),    # two cached tiles, then new rows; ragged last tile
    (1, 4, 129, 128, 257),    # capacity exactly Tk: the last tile's stores are clipped
    (3, 2, 512, 384, 1024),   # several units own new tiles; B > 1 (one rotary row per b)
])
def test_prefill_append_fused_matches_oracle_and_writes_cache(B, H, Tq, past, T_cap):
    """Prefill on a prefix of whole 128-key tiles with no kv_len: the attention kernel reads
    the new rows from their own buffers and the unit holding each new tile on its diagonal
    writes it into the caches."""
    wl, inp, cache, new = _case(B, H, Tq, past, T_cap, None, seed=24)
    d = to_device(inp)
    out = binding.mla_attn_append_fwd(d["q_nope"], d["q_pe"], new["k_nope"],
                                      new["k_pe_shared"], new["v"], cache["k_nope"],
                                      cache["k_pe_shared"], cache["v"], None, past,
                                      inp["softmax_scale"])
    torch.cuda.synchronize()
    assert_close(gpu_rows(out), oracle_for(inp), f"fused append B{B} H{H} Tq{Tq} past{past}")
    _check_cache(inp, cache, past, Tq, T_cap)
    # the same keys from one contiguous buffer give the same bits
    d["kv_len"] = None
    assert torch.equal(out.cpu(), run_gpu(d).cpu())


def test_decode_append_equals_attention_on_the_filled_cache():
    wl, inp, cache, new = _case(4, 8, 1, 511, 640, None, seed=22)
    d = to_device(inp)
    fused = binding.mla_attn_append_fwd(d["q_nope"], d["q_pe"], new["k_nope"],
                                        new["k_pe_shared"], new["v"], cache["k_nope"],
                                        cache["k_pe_shared"], cache["v"], d["kv_len"], 511,
                                        inp["softmax_scale"])
    plain = run_gpu(d)  # contiguous inputs holding prefix + new row
    assert torch.equal(fused.cpu(), plain.cpu())


def test_append_rejects_overflowing_cache():
    wl, inp, cache, new = _case(1, 2, 4, 10, 14, None, seed=23)
    d = to_device(inp)
    small = {k: v[..., :13, :] if k != "k_pe_shared" else v[:, :13].contiguous()
             for k, v in cache.items()}
    small = {k: v.contiguous() for k, v in small.items()}
    with pytest.raises(binding.MlaAttnError):
        binding.mla_attn_append_fwd(d["q_nope"], d["q_pe"], new["k_nope"], new["k_pe_shared"],
                                    new["v"], small["k_nope"], small["k_pe_shared"], small["v"],
                                    None, 10, inp["softmax_scale"])
