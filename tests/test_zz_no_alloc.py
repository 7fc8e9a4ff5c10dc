"""mla_attn_decode_noalloc: the decode call for callers that cannot allocate device memory.

Such callers (a server whose KV-cache pool owns all free HBM, a plugin inside a framework
whose allocator owns the device, a loop that cannot afford cudaMalloc's synchronisation)
get an entry point whose split-KV scratch is a fixed array inside the library.  These
tests call it through the C ABI and check each output against the fp64 oracle within the
parity tolerance, and bit for bit against mla_attn_fwd on the same inputs (both use the
same split plan and kernels).  Calls follow one another with different data and different
split plans, so each call finds an earlier call's partials, laid out for another plan, in
the shared array.  This file is named so that pytest collects it last.
"""
import ctypes

import pytest
import torch

from mla_causal_attention_gb300 import binding
from mla_causal_attention_gb300.inputs import make_inputs
from mla_causal_attention_gb300.workloads import WORKLOADS, Workload, softmax_scale_192
from gpu_helpers import assert_close, gpu_rows, oracle_for, run_gpu, to_device

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


def _check(inp, d, label):
    """One no-alloc call: within tolerance of the oracle and bit-equal to mla_attn_fwd."""
    want = run_gpu(d)
    got = torch.full_like(want, float("nan"))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert _noalloc(d, got, status) == 0
    assert int(status.item()) == 0
    assert_close(gpu_rows(got), oracle_for(inp), label)
    assert torch.equal(got, want), f"{label}: differs from mla_attn_fwd"


def _ragged_b8():
    return WORKLOADS["decode_ragged"].with_(B=8, past_len=2047, kv_len_range=(100, 2048))


@pytest.mark.parametrize("wl", [WORKLOADS["decode_p1000"], _ragged_b8()],
                         ids=["decode_p1000", "ragged_b8"])
def test_noalloc_matches_oracle_twice(wl):
    splits = binding.decode_plan(wl.B, wl.H, wl.Tk)[1]
    assert splits > 1  # these sizes really use the scratch array
    for seed in (11, 12):  # two calls in a row, different data
        inp = make_inputs(wl, seed=seed)
        _check(inp, to_device(inp), f"noalloc {wl.name} seed {seed}")


def test_noalloc_calls_with_changing_plans():
    """ragged_b8, then the page's decode shape, then ragged_b8 again: the partial layout in
    the shared array changes from call to call."""
    seq = [_ragged_b8(), WORKLOADS["decode_p1000"], _ragged_b8()]
    plans = [binding.decode_plan(w.B, w.H, w.Tk) for w in seq]
    assert plans[0] != plans[1]
    for k, wl in enumerate(seq):
        inp = make_inputs(wl, seed=20 + k)
        _check(inp, to_device(inp), f"noalloc sequence call {k} ({wl.name})")


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
