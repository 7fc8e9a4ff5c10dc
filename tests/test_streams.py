"""Calls launched on a stream other than the current one, each with a fresh workspace: the
workspace's zero fill is ordered before the call's kernels, and the result equals that of
the same call on the current stream."""
import pytest
import torch

from mla_causal_attention_gb300 import binding
from mla_causal_attention_gb300.inputs import make_inputs
from mla_causal_attention_gb300.workloads import Workload, softmax_scale_192
from gpu_helpers import run_gpu, to_device

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("B,H,Tq,past,kv", [
    (2, 8, 1, 299, (50, 300)),   # decode with several splits: partials in the workspace
    (1, 4, 200, 56, None),       # prefill
])
def test_side_stream_with_fresh_workspace(B, H, Tq, past, kv):
    inp = make_inputs(Workload("t", B, H, Tq, past, 1.0, kv, softmax_scale_192()), seed=21)
    d = to_device(inp)
    ref = run_gpu(d)
    side = torch.cuda.Stream()
    ws = binding.Workspace("cuda")
    out = torch.empty_like(ref)
    side.wait_stream(torch.cuda.current_stream())
    binding.mla_attn_fwd(d["q_nope"], d["q_pe"], d["k_nope"], d["k_pe_shared"], d["v"],
                         d["kv_len"], d["past_len"], d["softmax_scale"], out=out,
                         workspace=ws, stream=side)
    assert binding.mla_attn_get_status(ws, stream=side) == 0
    assert torch.equal(out, ref)
