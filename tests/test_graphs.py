"""CUDA graph capture of the library's calls.

A decode step (attention core, then the output projection), the latent-cache decode (three
kernels chained by programmatic dependent launches) and a chunked prefill are each captured
once and replayed with new inputs copied into the captured buffers.  Every replay must match
the same calls made eagerly, bit for bit (the kernels are deterministic), and the eager path
itself is checked against the oracle elsewhere.
"""
import pytest
import torch

from mla_causal_attention_gb300 import binding
from mla_causal_attention_gb300.inputs import make_inputs, make_latent_inputs, make_oproj_inputs
from mla_causal_attention_gb300.workloads import Workload, softmax_scale_192

pytestmark = pytest.mark.gpu


def _capture(fn):
    """Warm fn up eagerly on a side stream (allocations, tensor maps, kernel attributes),
    then capture it into a graph."""
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    with torch.cuda.graph(g):
        fn()
    torch.cuda.synchronize()
    return g


def _load(static, fresh):
    for k, t in fresh.items():
        if k in static and static[k] is not None:
            static[k].copy_(t)


def test_decode_step_with_oproj_replays():
    B, H, Tk = 4, 64, 700
    wl = Workload("g", B, H, 1, Tk - 1, 1.0, (100, Tk), softmax_scale_192())
    dev = torch.device("cuda")
    keys = ("q_nope", "q_pe", "k_nope", "k_pe_shared", "v", "kv_len")
    inp = make_inputs(wl, seed=1)
    st = {k: inp[k].to(dev) for k in keys}
    w = make_oproj_inputs(B, H, 1, 7168, seed=1)["w_o"].to(dev)
    out = torch.empty((B, H, 1, 128), dtype=torch.bfloat16, device=dev)
    y = torch.empty((B, 1, 7168), dtype=torch.bfloat16, device=dev)
    ws_a, ws_o = binding.Workspace(dev), binding.Workspace(dev)

    def step():
        binding.mla_attn_fwd(st["q_nope"], st["q_pe"], st["k_nope"], st["k_pe_shared"], st["v"],
                             st["kv_len"], inp["past_len"], inp["softmax_scale"], out=out,
                             workspace=ws_a)
        binding.mla_oproj_fwd(out, w, out=y, workspace=ws_o)

    g = _capture(step)
    for seed in (2, 3):
        fresh = make_inputs(wl, seed=seed)
        _load(st, {k: fresh[k].to(dev) for k in keys})
        g.replay()
        torch.cuda.synchronize()
        out_g, y_g = out.clone(), y.clone()
        step()
        torch.cuda.synchronize()
        assert torch.equal(out_g, out), seed
        assert torch.equal(y_g, y), seed
        assert bool(torch.isfinite(y.float()).all())


def test_latent_decode_replays():
    B, H, Tk = 6, 64, 1500
    wl = Workload("g", B, H, 1, Tk - 1, 1.0, (1, Tk), softmax_scale_192())
    dev = torch.device("cuda")
    keys = ("q_nope", "q_pe", "c_kv", "k_pe", "w_kvb", "kv_len")
    inp = make_latent_inputs(wl, seed=4)
    st = {k: inp[k].to(dev) for k in keys}
    out = torch.empty((B, H, 128), dtype=torch.bfloat16, device=dev)
    ws = binding.Workspace(dev)

    def step():
        binding.mla_latent_decode_fwd(st["q_nope"], st["q_pe"], st["c_kv"], st["k_pe"],
                                      st["w_kvb"], st["kv_len"], wl.softmax_scale, out=out,
                                      workspace=ws)

    g = _capture(step)
    for seed in (5, 6):
        fresh = make_latent_inputs(wl, seed=seed)
        _load(st, {k: fresh[k].to(dev) for k in keys})
        g.replay()
        torch.cuda.synchronize()
        out_g = out.clone()
        step()
        torch.cuda.synchronize()
        assert torch.equal(out_g, out), seed


def test_chunked_prefill_replays():
    B, H, Tq, past = 2, 4, 256, 512
    wl = Workload("g", B, H, Tq, past, 1.0, None, softmax_scale_192())
    dev = torch.device("cuda")
    keys = ("q_nope", "q_pe", "k_nope", "k_pe_shared", "v")
    inp = make_inputs(wl, seed=7)
    st = {k: inp[k].to(dev) for k in keys}
    out = torch.empty((B, H, Tq, 128), dtype=torch.bfloat16, device=dev)
    ws = binding.Workspace(dev)

    def step():
        binding.mla_attn_fwd(st["q_nope"], st["q_pe"], st["k_nope"], st["k_pe_shared"], st["v"],
                             None, past, inp["softmax_scale"], out=out, workspace=ws)

    g = _capture(step)
    for seed in (8, 9):
        fresh = make_inputs(wl, seed=seed)
        _load(st, {k: fresh[k].to(dev) for k in keys})
        g.replay()
        torch.cuda.synchronize()
        out_g = out.clone()
        step()
        torch.cuda.synchronize()
        assert torch.equal(out_g, out), seed
