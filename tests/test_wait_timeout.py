"""The bounded-wait paths of the kernels, exercised without any GPU fault.

Every wait inside the kernels is bounded: past its limit it records MLA_ERR_TIMEOUT in the
status word, raises a CTA-wide abort flag, waits (again bounded) for the CTA's own copies
and MMAs in flight, releases tensor memory and returns.  Test builds of the library (one
source compiled with a test-only define and a 2 ms wait limit; the library proper never
sets either) each withhold one plain release that starts no copy and carries no transaction
bytes:
  - prefill.cu, MLA_TEST_DROP_P_READY: one softmax warp of CTA 0 withholds one P-ready
    arrival, and the MMA warp's wait for it runs out;
  - decode.cu, MLA_TEST_DROP_SLOT_RELEASE: one consumer warp of the first CTA withholds its
    release of the first stage's slot, and the producer's wait to refill it runs out;
  - oproj.cu, MLA_TEST_DROP_STAGE_RELEASE: the MMA warp of CTA 0 skips the commit that
    releases its first stage, and the producers' waits to refill it run out;
  - latent.cu, MLA_TEST_DROP_SLOT_RELEASE: the MMA warp of CTA 0 skips the commit that
    releases latent slot 0 after its first tile, and the producer's wait to refill it runs
    out.
Each test checks that the call returns within a bounded time with the status word set to
MLA_ERR_TIMEOUT, and that the real library on the same GPU afterwards runs clean and matches
the oracle.
"""
import ctypes
import time

import numpy as np
import pytest
import torch

from mla_causal_attention_gb300 import binding
from mla_causal_attention_gb300.build import build_test_variant
from mla_causal_attention_gb300.inputs import make_inputs
from mla_causal_attention_gb300.workloads import Workload, softmax_scale_192
from gpu_helpers import assert_close, gpu_rows, oracle_for, run_gpu, to_device
from oracle import oracle_latent_rows, oracle_oproj_rows

pytestmark = pytest.mark.gpu


def _timeout_library(name="wait_timeout", source="prefill.cu", drop="MLA_TEST_DROP_P_READY"):
    path = build_test_variant(name, source, ["-DMLA_WAIT_LIMIT_NS=2000000ull", f"-D{drop}=1"])
    lib = ctypes.CDLL(path)
    p, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    lib.mla_attn_fwd.restype = i
    lib.mla_attn_fwd.argtypes = [p, p, p, p, p, p, i, i, i, i, i, f, p, p, sz, p]
    lib.mla_attn_get_status.restype = i
    lib.mla_attn_get_status.argtypes = [p, p]
    lib.mla_attn_workspace_bytes.restype = sz
    lib.mla_attn_workspace_bytes.argtypes = [i, i, i, i]
    lib.mla_oproj_workspace_bytes.restype = sz
    lib.mla_oproj_workspace_bytes.argtypes = []
    lib.mla_oproj_fwd.restype = i
    lib.mla_oproj_fwd.argtypes = [p, p, i, i, i, i, p, p, sz, p]
    lib.mla_latent_workspace_bytes.restype = sz
    lib.mla_latent_workspace_bytes.argtypes = [i, i, i]
    lib.mla_latent_decode_fwd.restype = i
    lib.mla_latent_decode_fwd.argtypes = [p, p, p, p, p, p, i, i, i, f, p, p, sz, p]
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


def test_decode_wait_gives_up_reports_timeout_and_device_stays_usable():
    # The page's decode shape: 64 heads over 1001 cached keys, 64-key splits of four 16-key
    # stages on a three-slot ring, so the producer of the first CTA waits to refill slot 0.
    w = Workload("timeout_decode", 1, 64, 1, 1000, 1.0, None, softmax_scale_192())
    inp = make_inputs(w, seed=32)
    d = to_device(inp)
    assert binding.decode_plan(1, 64, 1001) == (64, 16)
    lib = _timeout_library("wait_timeout_decode", "decode.cu", "MLA_TEST_DROP_SLOT_RELEASE")
    ws = torch.zeros(lib.mla_attn_workspace_bytes(1, 64, 1, 1001), dtype=torch.uint8,
                     device="cuda")
    out = torch.zeros((1, 64, 1, 128), dtype=torch.bfloat16, device="cuda")
    P = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    rc = lib.mla_attn_fwd(P(d["q_nope"]), P(d["q_pe"]), P(d["k_nope"]), P(d["k_pe_shared"]),
                          P(d["v"]), P(d["kv_len"]), 1, 64, 1, 1001, 1000,
                          ctypes.c_float(d["softmax_scale"]), P(out), P(ws),
                          ctypes.c_size_t(ws.numel()), stream)
    assert rc == 0
    st = lib.mla_attn_get_status(P(ws), stream)
    elapsed = time.perf_counter() - t0
    assert st == binding.MlaStatus.ERR_TIMEOUT, f"status {st}"
    assert elapsed < 5.0, f"the aborted launch took {elapsed:.2f} s"
    assert lib.mla_attn_get_status(P(ws), stream) == 0
    torch.cuda.synchronize()

    got = run_gpu(d)
    assert binding.mla_attn_get_status(device=torch.device("cuda")) == 0
    assert_close(gpu_rows(got), oracle_for(inp), "decode after a timed-out launch")


def test_oproj_wait_gives_up_reports_timeout_and_device_stays_usable():
    # The decode-width projection: 64 rows x 8192 -> 7168, one 48-column tile per CTA over
    # 128 k-blocks on a ten-stage ring, so the producers of CTA 0 wait to refill stage 0.
    B, H, T, N = 64, 64, 1, 7168
    g = torch.Generator().manual_seed(33)
    attn = torch.randn((B, H, T, 128), generator=g).to(torch.bfloat16)
    w = (torch.randn((N, H * 128), generator=g) * (H * 128) ** -0.5).to(torch.bfloat16)
    attn_d, w_d = attn.cuda(), w.cuda()
    lib = _timeout_library("wait_timeout_oproj", "oproj.cu", "MLA_TEST_DROP_STAGE_RELEASE")
    nb = lib.mla_oproj_workspace_bytes()
    ws = torch.zeros(nb, dtype=torch.uint8, device="cuda")
    y = torch.zeros((B, T, N), dtype=torch.bfloat16, device="cuda")
    P = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    rc = lib.mla_oproj_fwd(P(attn_d), P(w_d), B, H, T, N, P(y), P(ws), ctypes.c_size_t(nb),
                           stream)
    assert rc == 0
    st = lib.mla_attn_get_status(P(ws), stream)
    elapsed = time.perf_counter() - t0
    assert st == binding.MlaStatus.ERR_TIMEOUT, f"status {st}"
    assert elapsed < 5.0, f"the aborted launch took {elapsed:.2f} s"
    assert lib.mla_attn_get_status(P(ws), stream) == 0
    torch.cuda.synchronize()

    got = binding.mla_oproj_fwd(attn_d, w_d)
    torch.cuda.synchronize()
    rows = np.arange(0, B * T, 7)
    want = oracle_oproj_rows(attn, w, rows=rows)
    assert_close(got.float().cpu().numpy().reshape(B * T, N)[rows].astype(np.float64), want,
                 "o_proj after a timed-out launch")


def test_latent_wait_gives_up_reports_timeout_and_device_stays_usable():
    # 8 sequences of 8192 latent rows: 512 key tiles over the CTAs, several per CTA, so the
    # producer of CTA 0 waits to refill slot 0 for its second tile.
    B, H, Tk = 8, 64, 8192
    g = torch.Generator("cpu").manual_seed(34)
    mk = lambda *s: torch.randn(*s, generator=g).to(torch.bfloat16)  # noqa: E731
    h = dict(q_nope=mk(B, H, 128), q_pe=mk(B, H, 64), c_kv=mk(B, Tk, 512), k_pe=mk(B, Tk, 64),
             w_kvb=(torch.randn(H * 256, 512, generator=g) / 512 ** 0.5).to(torch.bfloat16))
    c = {k: v.cuda() for k, v in h.items()}
    lib = _timeout_library("wait_timeout_latent", "latent.cu", "MLA_TEST_DROP_SLOT_RELEASE")
    nb = lib.mla_latent_workspace_bytes(B, H, Tk)
    ws = torch.zeros(nb, dtype=torch.uint8, device="cuda")
    out = torch.zeros((B, H, 128), dtype=torch.bfloat16, device="cuda")
    P = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    scale = softmax_scale_192()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    rc = lib.mla_latent_decode_fwd(P(c["q_nope"]), P(c["q_pe"]), P(c["c_kv"]), P(c["k_pe"]),
                                   P(c["w_kvb"]), None, B, H, Tk, ctypes.c_float(scale),
                                   P(out), P(ws), ctypes.c_size_t(nb), stream)
    assert rc == 0
    st = lib.mla_attn_get_status(P(ws), stream)
    elapsed = time.perf_counter() - t0
    assert st == binding.MlaStatus.ERR_TIMEOUT, f"status {st}"
    assert elapsed < 5.0, f"the aborted launch took {elapsed:.2f} s"
    assert lib.mla_attn_get_status(P(ws), stream) == 0
    torch.cuda.synchronize()

    got = binding.mla_latent_decode_fwd(c["q_nope"], c["q_pe"], c["c_kv"], c["k_pe"],
                                        c["w_kvb"], None, scale)
    torch.cuda.synchronize()
    assert binding.mla_attn_get_status(device=got.device) == 0
    rows = np.arange(0, B * H, 5)
    want = oracle_latent_rows(h["q_nope"][:, :, None], h["q_pe"][:, :, None], h["c_kv"],
                              h["k_pe"], h["w_kvb"], None, Tk - 1, scale, rows=rows)
    assert_close(got.float().cpu().numpy().reshape(-1, 128)[rows], want,
                 "latent decode after a timed-out launch")
