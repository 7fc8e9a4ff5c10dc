"""Host side of the library's rotary step: YaRN frequencies computed by the library's own
host code (independent of the oracle's) agree with the oracle and with the page
configuration's split; bad configurations and sizes are refused before any launch."""
import ctypes
import math

import numpy as np
import pytest

from mla_causal_attention_gb300 import binding
from mla_causal_attention_gb300.build import build_library
from oracle import yarn

S = binding.MlaStatus
CONFIGS = [
    dict(theta=50000.0, factor=32.0, orig_max_pos=4096, beta_fast=1.0, beta_slow=1.0,
         mscale=1.0, mscale_all_dim=1.0),                       # the page's rope_scaling
    dict(theta=50000.0, factor=1.0, orig_max_pos=4096, beta_fast=32.0, beta_slow=1.0,
         mscale=1.0, mscale_all_dim=1.0),                       # no scaling
    dict(theta=10000.0, factor=40.0, orig_max_pos=4096, beta_fast=32.0, beta_slow=1.0,
         mscale=1.0, mscale_all_dim=0.707),                     # a wide ramp, ratio != 1
    dict(theta=1e6, factor=4.0, orig_max_pos=8192, beta_fast=5000.0, beta_slow=0.01,
         mscale=0.5, mscale_all_dim=2.0),                       # ramp clamped at both ends
]


@pytest.fixture(scope="module")
def lib():
    build_library()
    return binding.library()


def _cfg(c):
    return binding.RopeConfig(c["theta"], c["factor"], c["orig_max_pos"], c["beta_fast"],
                              c["beta_slow"], c["mscale"], c["mscale_all_dim"])


@pytest.mark.parametrize("c", CONFIGS)
def test_library_frequencies_match_oracle(lib, c):
    f_lib, m_lib = binding.mla_rope_frequencies(_cfg(c))
    f_or, m_or = yarn(**c)
    np.testing.assert_allclose(f_lib, f_or, rtol=1e-14, atol=0)
    assert m_lib == pytest.approx(m_or, rel=1e-14)


def test_page_configuration_split_in_library(lib):
    f, m = binding.mla_rope_frequencies(_cfg(CONFIGS[0]))
    plain = np.array([50000.0 ** (-2.0 * d / 64.0) for d in range(32)])
    np.testing.assert_allclose(f[:20], plain[:20], rtol=1e-15)
    np.testing.assert_allclose(f[20:], plain[20:] / 32.0, rtol=1e-15)
    assert m == 1.0


def test_default_binding_config_is_the_page_configuration(lib):
    f0, _ = binding.mla_rope_frequencies()
    f1, _ = binding.mla_rope_frequencies(_cfg(CONFIGS[0]))
    assert f0 == f1


@pytest.mark.parametrize("field,value", [("rope_theta", 1.0), ("factor", 0.5),
                                         ("original_max_position", 0.0),
                                         ("beta_slow", 0.0), ("beta_fast", 0.5),
                                         ("mscale", math.nan), ("factor", math.inf)])
def test_bad_configuration_is_refused(lib, field, value):
    cfg = _cfg(CONFIGS[0])
    setattr(cfg, field, value)
    f = (ctypes.c_double * 32)()
    m = ctypes.c_double()
    assert lib.mla_rope_frequencies(ctypes.byref(cfg), f, ctypes.byref(m)) == S.ERR_ARG
    assert lib.mla_rope_table(ctypes.byref(cfg), 16, ctypes.c_void_p(256), None) == S.ERR_ARG


def test_table_argument_errors(lib):
    cfg = _cfg(CONFIGS[0])
    assert lib.mla_rope_frequencies(None, None, None) == S.ERR_NULL
    assert lib.mla_rope_table(None, 16, ctypes.c_void_p(256), None) == S.ERR_NULL
    assert lib.mla_rope_table(ctypes.byref(cfg), 16, None, None) == S.ERR_NULL
    assert lib.mla_rope_table(ctypes.byref(cfg), 0, ctypes.c_void_p(256), None) == S.ERR_SHAPE
    assert lib.mla_rope_table(ctypes.byref(cfg), 16, ctypes.c_void_p(264), None) == S.ERR_ALIGN


def test_rope_workspace_bytes(lib):
    r256 = lambda x: -(-x // 256) * 256  # noqa: E731
    for B, H, Tq, Tk in [(1, 64, 16, 16), (3, 5, 1, 77), (64, 64, 1, 8192), (2, 3, 130, 207)]:
        base = binding.mla_attn_workspace_bytes(B, H, Tq, Tk)
        want = r256(base) + r256(B * H * Tq * 128) + r256(B * Tq * 128)
        assert lib.mla_attn_rope_workspace_bytes(B, H, Tq, Tk) == want
    assert lib.mla_attn_rope_workspace_bytes(0, 1, 1, 1) == 0
    assert lib.mla_attn_rope_workspace_bytes(1, 1, 2, 1) == 0


def _rope_call(lib, P, B=1, H=1, Tq=2, T_cap=4, past=1, scale=0.1, table_rows=8, ws=1 << 16,
               kvl=None, **over):
    args = dict(q=P[0], qr=P[1], kn=P[2], kr=P[3], v=P[4], kc=P[5], krc=P[6], vc=P[7],
                table=P[8], out=P[9], wsp=P[10])
    args.update(over)
    return lib.mla_attn_rope_append_fwd(args["q"], args["qr"], args["kn"], args["kr"],
                                        args["v"], args["kc"], args["krc"], args["vc"], kvl, B,
                                        H, Tq, T_cap, past, scale, args["table"], table_rows,
                                        args["out"], args["wsp"], ws, None)


def test_rope_append_host_errors_before_any_launch(lib):
    buf = (ctypes.c_uint8 * 8192)()
    base = (ctypes.addressof(buf) + 255) & ~255
    P = [ctypes.c_void_p(base + 256 * i) for i in range(11)]
    for k in ("qr", "kn", "kr", "v", "kc", "krc", "vc", "table", "q", "out"):
        assert _rope_call(lib, P, **{k: None}) == S.ERR_NULL, k
    assert _rope_call(lib, P, T_cap=2) == S.ERR_SHAPE          # past + Tq > T_cap
    assert _rope_call(lib, P, table_rows=2) == S.ERR_SHAPE     # table shorter than Tk
    assert _rope_call(lib, P, past=-1) == S.ERR_SHAPE
    assert _rope_call(lib, P, table=ctypes.c_void_p(base + 4)) == S.ERR_ALIGN
    assert _rope_call(lib, P, kc=ctypes.c_void_p(base + 8)) == S.ERR_ALIGN
    assert _rope_call(lib, P, ws=256) == S.ERR_WORKSPACE
    assert _rope_call(lib, P, wsp=None) == S.ERR_WORKSPACE
    assert _rope_call(lib, P, scale=-1.0) == S.ERR_ARG
    import torch
    if not torch.cuda.is_available():
        assert _rope_call(lib, P) in (S.ERR_CUDA, S.ERR_DEVICE)
        assert _rope_call(lib, P, Tq=1, past=3) in (S.ERR_CUDA, S.ERR_DEVICE)
