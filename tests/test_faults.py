"""Device-detected problems reach the status word without faulting the GPU."""
import pytest
import torch

from mla_causal_attention_gb300 import binding
from mla_causal_attention_gb300.inputs import make_inputs
from mla_causal_attention_gb300.workloads import Workload, softmax_scale_192
from gpu_helpers import run_gpu, to_device

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("Tq,past", [(1, 99), (64, 36)])
@pytest.mark.parametrize("bad", [0, 101, -5])
def test_out_of_range_kv_len_sets_status(Tq, past, bad):
    w = Workload("t", 2, 4, Tq, past, 1.0, None, softmax_scale_192())
    inp = make_inputs(w, seed=0)
    ws = binding.Workspace("cuda")
    d = to_device(inp)
    assert binding.mla_attn_get_status(ws) == 0
    d["kv_len"][1] = bad
    from mla_causal_attention_gb300 import mla_attn_fwd
    out = mla_attn_fwd(d["q_nope"], d["q_pe"], d["k_nope"], d["k_pe_shared"], d["v"],
                       d["kv_len"], d["past_len"], d["softmax_scale"], workspace=ws)
    assert binding.mla_attn_get_status(ws) == binding.MlaStatus.ERR_KVLEN
    assert binding.mla_attn_get_status(ws) == 0  # reading clears it
    assert torch.isfinite(out.float()).all()
    # the library stays usable afterwards
    d["kv_len"][1] = w.Tk
    run_gpu(d)
    assert binding.mla_attn_get_status(ws) == 0


def test_host_errors_raise():
    w = Workload("t", 1, 2, 4, 0, 1.0, None, softmax_scale_192())
    d = to_device(make_inputs(w, seed=0))
    from mla_causal_attention_gb300 import mla_attn_fwd
    with pytest.raises(binding.MlaAttnError):
        mla_attn_fwd(d["q_nope"], d["q_pe"], d["k_nope"], d["k_pe_shared"], d["v"],
                     d["kv_len"], 1, d["softmax_scale"])  # past_len inconsistent with Tk
    with pytest.raises(binding.MlaAttnError):
        mla_attn_fwd(d["q_nope"], d["q_pe"], d["k_nope"], d["k_pe_shared"], d["v"],
                     d["kv_len"], 0, -1.0)


@pytest.mark.parametrize("bad", [0, 301, -5])
def test_latent_out_of_range_kv_len_sets_status(bad):
    """The latent path clamps kv_len into [1, Tk] for its partition and reports the bad value."""
    from mla_causal_attention_gb300.inputs import make_latent_inputs
    w = Workload("t", 3, 64, 1, 299, 1.0, (1, 300), softmax_scale_192())
    inp = make_latent_inputs(w, seed=3)
    d = {k: v.cuda() for k, v in inp.items()}
    ws = binding.Workspace("cuda")
    d["kv_len"][1] = bad

    def call():
        return binding.mla_latent_decode_fwd(d["q_nope"], d["q_pe"], d["c_kv"], d["k_pe"],
                                             d["w_kvb"], d["kv_len"], w.softmax_scale,
                                             workspace=ws)
    out = call()
    assert binding.mla_attn_get_status(ws) == binding.MlaStatus.ERR_KVLEN
    assert binding.mla_attn_get_status(ws) == 0  # reading clears it
    assert torch.isfinite(out.float()).all()
    d["kv_len"][1] = 300
    call()
    assert binding.mla_attn_get_status(ws) == 0
