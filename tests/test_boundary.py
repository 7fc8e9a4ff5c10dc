"""The C-ABI library: builds, loads, exports every declared symbol, rejects bad arguments
on the host before touching a GPU.  No kernel is launched here."""
import ctypes
import os
import re

import pytest

from mla_causal_attention_gb300 import binding
from mla_causal_attention_gb300.build import build_library

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build_library()
    return binding.library()


def declared_functions():
    names = []
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            names += re.findall(r"MLA_API\s+[\w\s\*]+?\b(\w+)\s*\(", src)
    return sorted(set(names))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert "mla_attn_fwd" in names and "mla_attn_get_status" in names
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/ but not exported"
    assert set(binding.EXPORTED) <= set(names)


def test_status_strings(lib):
    for code in range(10):
        s = lib.mla_status_string(code).decode()
        assert s.startswith("MLA_")
    assert lib.mla_status_string(99).decode() == "unknown mla_status"


def test_workspace_sizes(lib):
    assert binding.mla_attn_workspace_bytes(1, 64, 16, 16) == 256
    assert binding.mla_attn_workspace_bytes(0, 64, 1, 1) == 0
    assert binding.mla_attn_workspace_bytes(1, 1, 2, 1) == 0
    # decode: status word + per-(b, h, split) (max, sum, 128 accumulators) in fp32
    c, s = binding.decode_plan(64, 64, 8192)
    assert c % 64 == 0 and s == -(-8192 // c)
    ml = -(-(64 * 64 * s * 8) // 256) * 256
    want = 256 if s == 1 else 256 + ml + 64 * 64 * s * 128 * 4
    assert binding.mla_attn_workspace_bytes(64, 64, 1, 8192) == want


def test_workspace_keeps_accumulators_16_byte_aligned(lib):
    # an odd number of (b, h, split) partials must not misalign the accumulator array
    for B, H, Tk in [(1, 1, 200), (3, 5, 77), (1, 3, 1000)]:
        c, s = binding.decode_plan(B, H, Tk)
        n = binding.mla_attn_workspace_bytes(B, H, 1, Tk)
        if s > 1:
            assert (n - 256 - B * H * s * 512) % 256 == 0


def test_decode_plan_is_sane(lib):
    for B, H, Tk in [(1, 64, 1001), (64, 64, 8192), (3, 5, 17), (1, 1, 1)]:
        c, s = binding.decode_plan(B, H, Tk)
        assert 32 <= c <= 1024 and c % 32 == 0
        assert (s - 1) * c < Tk <= s * c
    import torch
    if not torch.cuda.is_available():  # the plan assumes GB300's 152 SMs without a device
        # one sequence of 64 heads is smaller than a wave: about 2 CTAs per SM
        assert binding.decode_plan(1, 64, 1001) == (64, 16)
        assert binding.decode_plan(64, 64, 8192) == (1024, 8)


def _call(lib, ptrs, B=1, H=1, Tq=2, Tk=2, past=0, scale=0.1, ws=256, opts=None):
    q, qr, k, kr, v, kvl, out, wsp = ptrs
    f = lib.mla_attn_fwd_ex if opts is not None else lib.mla_attn_fwd
    args = [q, qr, k, kr, v, kvl, B, H, Tq, Tk, past, scale, out, wsp, ws, None]
    if opts is not None:
        args.append(ctypes.byref(opts))
    return f(*args)


def test_host_side_errors_before_any_launch(lib):
    buf = (ctypes.c_uint8 * 4096)()
    base = (ctypes.addressof(buf) + 255) & ~255
    P = [ctypes.c_void_p(base + 256 * i) for i in range(8)]
    S = binding.MlaStatus
    ok_ptrs = P[:5] + [None] + P[6:]
    assert _call(lib, [None] + ok_ptrs[1:]) == S.ERR_NULL
    assert _call(lib, ok_ptrs[:6] + [None, P[7]]) == S.ERR_NULL
    assert _call(lib, ok_ptrs[:7] + [None]) == S.ERR_WORKSPACE
    assert _call(lib, ok_ptrs, Tk=3) == S.ERR_SHAPE          # Tk != past_len + Tq
    assert _call(lib, ok_ptrs, B=0) == S.ERR_SHAPE
    assert _call(lib, ok_ptrs, past=-1, Tk=1) == S.ERR_SHAPE
    assert _call(lib, ok_ptrs, Tq=0, Tk=0) == S.ERR_SHAPE
    bad = list(ok_ptrs)
    bad[2] = ctypes.c_void_p(base + 8)
    assert _call(lib, bad) == S.ERR_ALIGN
    assert _call(lib, ok_ptrs, scale=0.0) == S.ERR_ARG
    assert _call(lib, ok_ptrs, scale=float("nan")) == S.ERR_ARG
    o = binding._Options(7, 0)
    assert _call(lib, ok_ptrs, opts=o) == S.ERR_ARG
    o = binding._Options(binding.PATH_DECODE, 0)
    assert _call(lib, ok_ptrs, opts=o) == S.ERR_ARG         # decode path needs Tq == 1
    # Valid arguments on a machine without an sm_103 GPU fail cleanly on the device check.
    import torch
    if not torch.cuda.is_available():
        assert _call(lib, ok_ptrs) in (S.ERR_CUDA, S.ERR_DEVICE)


def test_binding_refuses_cpu_tensors(lib):
    import torch
    x = torch.zeros(1, 1, 2, 128, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        binding.mla_attn_fwd(x, x, x, x, x, None, 0, 0.1)


def test_masked_entry_host_errors(lib):
    buf = (ctypes.c_uint8 * 4096)()
    base = (ctypes.addressof(buf) + 255) & ~255
    P = [ctypes.c_void_p(base + 256 * i) for i in range(9)]
    S = binding.MlaStatus
    q, qr, k, kr, v, km, out, ws = P[:8]
    call = lambda km_, B=1, Tq=2, Tk=2, past=0, wsb=4096: lib.mla_attn_masked_fwd(  # noqa
        q, qr, k, kr, v, None, km_, B, 1, Tq, Tk, past, 0.1, out, ws, wsb, None)
    assert call(None) == S.ERR_NULL
    assert call(km, Tk=3) == S.ERR_SHAPE
    import torch
    # prefill needs room for the packed mask (checked after the device check)
    want = (S.ERR_WORKSPACE,) if torch.cuda.is_available() else (S.ERR_CUDA, S.ERR_DEVICE)
    assert call(km, wsb=256) in want
    assert lib.mla_attn_masked_workspace_bytes(2, 4, 130, 207) == 256 + 256
    assert lib.mla_attn_masked_workspace_bytes(3, 8, 1, 300) == \
        lib.mla_attn_workspace_bytes(3, 8, 1, 300)
    if not torch.cuda.is_available():
        assert call(km) in (S.ERR_CUDA, S.ERR_DEVICE)


def test_oproj_host_errors(lib):
    """mla_oproj_fwd rejects bad arguments before any device work."""
    buf = ctypes.create_string_buffer(1 << 16)
    base = (ctypes.addressof(buf) + 255) & ~255
    p = lambda off=0: ctypes.c_void_p(base + off)  # noqa: E731
    ws, n = p(), 256
    assert lib.mla_oproj_workspace_bytes() == 256
    # null pointers
    assert lib.mla_oproj_fwd(None, p(), 1, 1, 1, 32, p(), ws, n, None) == binding.MlaStatus.ERR_NULL
    assert lib.mla_oproj_fwd(p(), p(), 1, 1, 1, 32, None, ws, n, None) == binding.MlaStatus.ERR_NULL
    # sizes: N a multiple of 32, every size >= 1
    for B, H, T, N in [(0, 1, 1, 32), (1, 0, 1, 32), (1, 1, 0, 32), (1, 1, 1, 48), (1, 1, 1, 0)]:
        assert lib.mla_oproj_fwd(p(), p(), B, H, T, N, p(), ws, n, None) == \
            binding.MlaStatus.ERR_SHAPE, (B, H, T, N)
    # alignment and workspace
    assert lib.mla_oproj_fwd(p(8), p(), 1, 1, 1, 32, p(), ws, n, None) == binding.MlaStatus.ERR_ALIGN
    assert lib.mla_oproj_fwd(p(), p(), 1, 1, 1, 32, p(), None, n, None) == \
        binding.MlaStatus.ERR_WORKSPACE
    assert lib.mla_oproj_fwd(p(), p(), 1, 1, 1, 32, p(), ws, 8, None) == \
        binding.MlaStatus.ERR_WORKSPACE
