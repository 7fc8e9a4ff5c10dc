"""The bounded-wait path of the prefill kernel, exercised without any GPU fault.

Every wait inside the kernels is bounded: past its limit it records MLA_ERR_TIMEOUT in the
status word, raises a CTA-wide abort flag, waits (again bounded) for the CTA's own copies
and MMAs in flight, releases tensor memory and returns.  A test build of the library
(prefill.cu compiled with MLA_TEST_DROP_P_READY and a 2 ms wait limit; the library proper
never sets either) has one softmax warp of CTA 0 withhold one P-ready arrival, a plain
mbarrier arrive that starts no copy and carries no transaction bytes.  The MMA warp's wait
for it runs out.  The test checks that the call returns within a bounded time with the
status word set to MLA_ERR_TIMEOUT, and that the real library on the same GPU afterwards
runs clean and matches the oracle.
"""
import ctypes
import time

import pytest
import torch

from mla_causal_attention_gb300 import binding
from mla_causal_attention_gb300.build import build_test_variant
from mla_causal_attention_gb300.inputs import make_inputs
from mla_causal_attention_gb300.workloads import Workload, softmax_scale_192
from gpu_helpers import assert_close, gpu_rows, oracle_for, run_gpu, to_device

pytestmark = pytest.mark.gpu


def _timeout_library():
    path = build_test_variant("wait_timeout", "prefill.cu",
                              ["-DMLA_WAIT_LIMIT_NS=2000000ull", "-DMLA_TEST_DROP_P_READY=1"])
    lib = ctypes.CDLL(path)
    p, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    lib.mla_attn_fwd.restype = i
    lib.mla_attn_fwd.argtypes = [p, p, p, p, p, p, i, i, i, i, i, f, p, p, sz, p]
    lib.mla_attn_get_status.restype = i
    lib.mla_attn_get_status.argtypes = [p, p]
    return lib


def test_prefill_wait_gives_up_reports_timeout_and_device_stays_usable():
    # 2 heads x 512 queries: 4 units on 4 CTAs; CTA 0's first unit (the last query-tile pair
    # of head 0) has 3 key tiles in its first query tile, so the withheld arrival on its
    # second key tile is one the MMA warp waits for.
    w = Workload("timeout", 1, 2, 512, 0, 1.0, None, softmax_scale_192())
    inp = make_inputs(w, seed=31)
    d = to_device(inp)
    lib = _timeout_library()
    ws = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    out = torch.zeros((1, 2, 512, 128), dtype=torch.bfloat16, device="cuda")
    P = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    rc = lib.mla_attn_fwd(P(d["q_nope"]), P(d["q_pe"]), P(d["k_nope"]), P(d["k_pe_shared"]),
                          P(d["v"]), P(d["kv_len"]), 1, 2, 512, 512, 0,
                          ctypes.c_float(d["softmax_scale"]), P(out), P(ws),
                          ctypes.c_size_t(ws.numel()), stream)
    assert rc == 0
    st = lib.mla_attn_get_status(P(ws), stream)  # synchronises the stream
    elapsed = time.perf_counter() - t0
    assert st == binding.MlaStatus.ERR_TIMEOUT, f"status {st}"
    assert elapsed < 5.0, f"the aborted launch took {elapsed:.2f} s"
    # The status word was read and cleared; nothing else is pending on the stream.
    assert lib.mla_attn_get_status(P(ws), stream) == 0
    torch.cuda.synchronize()

    # The library proper on the same GPU and inputs: clean status, oracle parity.
    got = run_gpu(d)
    assert binding.mla_attn_get_status(device=torch.device("cuda")) == 0
    assert_close(gpu_rows(got), oracle_for(inp), "prefill after a timed-out launch")
