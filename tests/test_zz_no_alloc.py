"""mla_attn_decode_noalloc: the decode call for callers that cannot allocate device memory.

Such callers (a server whose KV-cache pool owns all free HBM, a plugin inside a framework
whose allocator owns the device, a loop that cannot afford cudaMalloc's synchronisation)
get an entry point whose split-KV scratch is a fixed array inside the library.  These
tests call it through the C ABI and check it against mla_attn_fwd on the same inputs,
twice in a row (the second call finds the first call's partials in the shared array).
This file is named so that pytest collects it last.
"""
import ctypes

import numpy as np
import pytest
import torch

from mla_causal_attention_gb300 import binding
from mla_causal_attention_gb300.inputs import make_inputs
from mla_causal_attention_gb300.workloads import WORKLOADS, Workload, softmax_scale_192
from gpu_helpers import MAX_ABS_TOL, MEAN_ABS_TOL, run_gpu, to_device

pytestmark = pytest.mark.gpu


def _lib():
    lib = binding.library()
    f = lib.mla_attn_decode_noalloc
    p = ctypes.c_void_p
    f.restype = ctypes.c_int
    f.argtypes = [p, p, p, p, p, p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_float,
                  p, p, p]
    return f


def _noalloc(d, out, status=None):
    f = _lib()
    B, H, _, _ = d["q_nope"].shape
    Tk = d["k_nope"].shape[2]
    ptr = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())  # noqa: E731
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = f(ptr(d["q_nope"]), ptr(d["q_pe"]), ptr(d["k_nope"]), ptr(d["k_pe_shared"]),
           ptr(d["v"]), ptr(d["kv_len"]), B, H, Tk, float(d["softmax_scale"]), ptr(out),
           ptr(status), stream)
    torch.cuda.synchronize()
    return rc


def _compare(a, b):
    e = (a.double() - b.double()).abs()
    assert torch.isfinite(a.float()).all()
    assert e.max().item() <= MAX_ABS_TOL and e.mean().item() <= MEAN_ABS_TOL


def _cases():
    ragged = WORKLOADS["decode_ragged"].with_(B=8, past_len=2047, kv_len_range=(100, 2048))
    return [WORKLOADS["decode_p1000"], ragged]


@pytest.mark.parametrize("wl", _cases(), ids=["decode_p1000", "ragged_b8"])
def test_noalloc_matches_fwd_twice(wl):
    splits = binding.decode_plan(wl.B, wl.H, wl.Tk)[1]
    assert splits > 1  # these sizes really use the scratch array
    first = to_device(make_inputs(wl, seed=11))
    second = to_device(make_inputs(wl, seed=12))
    for d in (first, second):  # two calls in a row, different data
        want = run_gpu(d)
        got = torch.empty_like(want)
        assert _noalloc(d, got) == 0
        _compare(got, want)


def test_noalloc_reports_kv_len_errors_and_rejects_oversized_plans():
    wl = Workload("t", 2, 4, 1, 299, 1.0, None, softmax_scale_192())
    d = to_device(make_inputs(wl, seed=13))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.empty((2, 4, 1, 128), dtype=torch.bfloat16, device="cuda")
    d["kv_len"][0] = 0
    assert _noalloc(d, out, status) == 0
    assert int(status.item()) == binding.MlaStatus.ERR_KVLEN
    # 64 x 64 heads over 262144 cached keys would need more partials than the array holds;
    # the call is refused before anything is launched.
    f = _lib()
    dummy = ctypes.c_void_p(d["k_nope"].data_ptr())
    rc = f(dummy, dummy, dummy, dummy, dummy, None, 64, 64, 262144, 0.07, dummy, None, None)
    assert rc == binding.MlaStatus.ERR_WORKSPACE
