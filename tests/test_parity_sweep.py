"""Seeded random sweep of sizes through the public calls, every output row against the oracle.

The fixed-shape parity tests pin the configurations and the chosen edge cases.  This sweep
draws the sizes themselves from a fixed seed: head counts that are not multiples of the
decode kernel's 4-head groups, past lengths that are not multiples of 128, query counts
from 2 to 600 (ragged last query tiles, units whose second tile is empty or partial),
kv_len ragged per sequence or absent, 2D key masks with left padding and holes, and cache
appends into caches of random capacity (half the prefills on a prefix of whole key tiles,
where the append happens inside the attention kernel).  Every case is small enough for the
oracle to compute all rows in well under a second, and each runs through mla_attn_fwd
(prefill or decode path chosen by Tq), mla_attn_masked_fwd or mla_attn_append_fwd.
"""
import numpy as np
import pytest
import torch

from mla_causal_attention_gb300 import binding
from mla_causal_attention_gb300.inputs import make_inputs
from mla_causal_attention_gb300.workloads import Workload, softmax_scale_192
from gpu_helpers import assert_close, gpu_rows, oracle_for, run_gpu, to_device
from oracle import oracle_rows

pytestmark = pytest.mark.gpu


def _draw_cases(seed, n, decode):
    rng = np.random.default_rng(seed)
    cases = []
    for k in range(n):
        B = int(rng.integers(1, 4 if not decode else 10))
        H = int(rng.integers(1, 8 if not decode else 12))
        Tq = 1 if decode else int(rng.integers(2, 601))
        past = int(rng.integers(0, 1500 if not decode else 6000))
        if decode:
            past = max(past, 0)
        Tk = past + Tq
        kv = None
        if rng.random() < 0.5:
            lo = int(rng.integers(1, Tk + 1))
            kv = (lo, Tk)
        cases.append((k, B, H, Tq, past, kv))
    return cases


def _ids(cases):
    return [f"B{B}_H{H}_Tq{Tq}_p{p}_kv{'-' if kv is None else kv[0]}" for _, B, H, Tq, p, kv in cases]


PREFILL = _draw_cases(2026, 20, decode=False)
DECODE = _draw_cases(2027, 20, decode=True)


@pytest.mark.parametrize("k,B,H,Tq,past,kv", PREFILL, ids=_ids(PREFILL))
def test_prefill_sweep_every_row(k, B, H, Tq, past, kv):
    w = Workload(f"sweep_p{k}", B, H, Tq, past, 1.0, kv, softmax_scale_192())
    inp = make_inputs(w, seed=100 + k)
    got = run_gpu(to_device(inp))
    assert binding.mla_attn_get_status(device=got.device) == 0
    assert_close(gpu_rows(got), oracle_for(inp), f"prefill sweep {k}")


@pytest.mark.parametrize("k,B,H,Tq,past,kv", DECODE, ids=_ids(DECODE))
def test_decode_sweep_every_row(k, B, H, Tq, past, kv):
    w = Workload(f"sweep_d{k}", B, H, Tq, past, 1.0, kv, softmax_scale_192())
    inp = make_inputs(w, seed=200 + k)
    got = run_gpu(to_device(inp))
    assert binding.mla_attn_get_status(device=got.device) == 0
    assert_close(gpu_rows(got), oracle_for(inp), f"decode sweep {k}")


MASKED = _draw_cases(2028, 6, decode=False)[:3] + _draw_cases(2029, 6, decode=True)[:3]


@pytest.mark.parametrize("k,B,H,Tq,past,kv", MASKED, ids=_ids(MASKED))
def test_masked_sweep_every_row(k, B, H, Tq, past, kv):
    w = Workload(f"sweep_m{k}", B, H, Tq, past, 1.0, kv, softmax_scale_192())
    inp = make_inputs(w, seed=300 + k + 17 * Tq)
    rng = np.random.default_rng(400 + k)
    Tk = past + Tq
    mask = np.ones((B, Tk), dtype=np.uint8)
    for b in range(B):
        mask[b, : int(rng.integers(0, max(1, Tk // 3)))] = 0
    mask &= (rng.random((B, Tk)) > 0.2).astype(np.uint8)
    d = to_device(inp)
    out = binding.mla_attn_masked_fwd(d["q_nope"], d["q_pe"], d["k_nope"], d["k_pe_shared"],
                                      d["v"], d["kv_len"], torch.from_numpy(mask).cuda(),
                                      inp["past_len"], inp["softmax_scale"])
    torch.cuda.synchronize()
    assert binding.mla_attn_get_status(device=out.device) == 0
    want = oracle_rows(inp["q_nope"], inp["q_pe"], inp["k_nope"], inp["k_pe_shared"],
                       inp["v"], inp["kv_len"], inp["past_len"], inp["softmax_scale"],
                       key_mask=mask)
    assert_close(gpu_rows(out), want, f"masked sweep {k}")


def _append_cases(seed, n):
    rng = np.random.default_rng(seed)
    cases = []
    for k in range(n):
        B = int(rng.integers(1, 4))
        H = int(rng.integers(1, 7))
        Tq = int(rng.integers(2, 500)) if k % 3 else 1
        if Tq > 1 and k % 2 == 0:
            past = 128 * int(rng.integers(0, 8))  # whole key tiles: the fused path
        else:
            past = int(rng.integers(0, 1200))
        spare = int(rng.integers(0, 300))
        cases.append((k, B, H, Tq, past, past + Tq + spare))
    return cases


APPEND = _append_cases(2030, 10)


@pytest.mark.parametrize("k,B,H,Tq,past,T_cap", APPEND,
                         ids=[f"B{B}_H{H}_Tq{Tq}_p{p}_cap{c}" for _, B, H, Tq, p, c in APPEND])
def test_append_sweep_every_row_and_cache(k, B, H, Tq, past, T_cap):
    """mla_attn_append_fwd on seeded random sizes: half the prefills on a prefix of whole key
    tiles (the append inside the attention kernel), the rest copy first; decode rows too.
    The output matches the oracle over the concatenated keys; the caches hold exactly the
    prefix and the new rows, every later row untouched."""
    poison = 3.0
    w = Workload(f"sweep_a{k}", B, H, Tq, past, 1.0, None, softmax_scale_192())
    inp = make_inputs(w, seed=500 + k)
    Tk = past + Tq
    cache = {}
    for name, shape in (("k_nope", (B, H, T_cap, 128)), ("v", (B, H, T_cap, 128)),
                        ("k_pe_shared", (B, T_cap, 64))):
        c = torch.full(shape, poison, dtype=torch.bfloat16)
        if name == "k_pe_shared":
            c[:, :past] = inp[name][:, :past]
        else:
            c[:, :, :past] = inp[name][:, :, :past]
        cache[name] = c.cuda()
    new = {"k_nope": inp["k_nope"][:, :, past:Tk].contiguous().cuda(),
           "v": inp["v"][:, :, past:Tk].contiguous().cuda(),
           "k_pe_shared": inp["k_pe_shared"][:, past:Tk].contiguous().cuda()}
    d = to_device(inp)
    out = binding.mla_attn_append_fwd(d["q_nope"], d["q_pe"], new["k_nope"],
                                      new["k_pe_shared"], new["v"], cache["k_nope"],
                                      cache["k_pe_shared"], cache["v"], None, past,
                                      inp["softmax_scale"])
    torch.cuda.synchronize()
    assert binding.mla_attn_get_status(device=out.device) == 0
    assert_close(gpu_rows(out), oracle_for(inp), f"append sweep {k}")
    for name in ("k_nope", "v"):
        c = cache[name].cpu()
        assert torch.equal(c[:, :, :Tk], inp[name]), name
        assert bool((c[:, :, Tk:] == poison).all()), name
    c = cache["k_pe_shared"].cpu()
    assert torch.equal(c[:, :Tk], inp["k_pe_shared"])
    assert bool((c[:, Tk:] == poison).all())
