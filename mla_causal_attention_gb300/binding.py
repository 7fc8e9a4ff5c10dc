"""ctypes binding of libmla_attn.so (argument marshalling only).

Every step of the attention core runs in the library's CUDA kernels; this module only
checks tensor dtypes/devices, passes raw device pointers, sizes and the current CUDA
stream, and turns status codes into exceptions.  There is no fallback: if the library is
missing, every call raises.
"""
from __future__ import annotations

import ctypes
import enum
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libmla_attn.so")
_lock = threading.Lock()
_lib = None


class MlaStatus(enum.IntEnum):
    OK = 0
    ERR_NULL = 1
    ERR_SHAPE = 2
    ERR_ALIGN = 3
    ERR_WORKSPACE = 4
    ERR_DEVICE = 5
    ERR_CUDA = 6
    ERR_KVLEN = 7
    ERR_TIMEOUT = 8
    ERR_ARG = 9


PATH_AUTO, PATH_PREFILL, PATH_DECODE = 0, 1, 2


class MlaAttnError(RuntimeError):
    def __init__(self, status: int, msg: str = ""):
        self.status = MlaStatus(status) if status in MlaStatus._value2member_map_ else status
        super().__init__(f"{msg}{self.status!r}: {_status_string(status)}")


class RopeConfig(ctypes.Structure):
    """mla_rope_config: YaRN rotary scaling (Kimi K2's values are the defaults)."""
    _fields_ = [("rope_theta", ctypes.c_double), ("factor", ctypes.c_double),
                ("original_max_position", ctypes.c_double), ("beta_fast", ctypes.c_double),
                ("beta_slow", ctypes.c_double), ("mscale", ctypes.c_double),
                ("mscale_all_dim", ctypes.c_double)]

    def __init__(self, rope_theta=50000.0, factor=32.0, original_max_position=4096,
                 beta_fast=1.0, beta_slow=1.0, mscale=1.0, mscale_all_dim=1.0):
        super().__init__(float(rope_theta), float(factor), float(original_max_position),
                         float(beta_fast), float(beta_slow), float(mscale),
                         float(mscale_all_dim))


class _Options(ctypes.Structure):
    _fields_ = [("path", ctypes.c_int), ("decode_chunk", ctypes.c_int),
                ("reserved", ctypes.c_int * 6)]


EXPORTED = ("mla_attn_workspace_bytes", "mla_attn_fwd", "mla_attn_fwd_ex",
            "mla_attn_get_status", "mla_status_string", "mla_attn_decode_plan",
            "mla_attn_append_fwd", "mla_rope_frequencies", "mla_rope_table",
            "mla_attn_rope_workspace_bytes", "mla_attn_rope_append_fwd",
            "mla_attn_masked_workspace_bytes", "mla_attn_masked_fwd",
            "mla_latent_workspace_bytes", "mla_latent_decode_fwd",
            "mla_oproj_workspace_bytes", "mla_oproj_fwd")


def library():
    """Load libmla_attn.so (built in-tree by build.py); raise if it is not there."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise MlaAttnError(MlaStatus.ERR_CUDA,
                               f"{LIB_PATH} is not built (run python -m "
                               "mla_causal_attention_gb300.build); ")
        lib = ctypes.CDLL(LIB_PATH)
        p, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        fwd_args = [p, p, p, p, p, p, i, i, i, i, i, f, p, p, sz, p]
        lib.mla_attn_workspace_bytes.restype = sz
        lib.mla_attn_workspace_bytes.argtypes = [i, i, i, i]
        lib.mla_attn_fwd.restype = i
        lib.mla_attn_fwd.argtypes = fwd_args
        lib.mla_attn_fwd_ex.restype = i
        lib.mla_attn_fwd_ex.argtypes = fwd_args + [ctypes.POINTER(_Options)]
        lib.mla_attn_get_status.restype = i
        lib.mla_attn_get_status.argtypes = [p, p]
        lib.mla_status_string.restype = ctypes.c_char_p
        lib.mla_status_string.argtypes = [i]
        lib.mla_attn_decode_plan.restype = i
        lib.mla_attn_decode_plan.argtypes = [i, i, i, ctypes.POINTER(i), ctypes.POINTER(i)]
        lib.mla_attn_append_fwd.restype = i
        lib.mla_attn_append_fwd.argtypes = [p, p, p, p, p, p, p, p, p, i, i, i, i, i, f, p, p,
                                            sz, p]
        lib.mla_attn_masked_workspace_bytes.restype = sz
        lib.mla_attn_masked_workspace_bytes.argtypes = [i, i, i, i]
        lib.mla_attn_masked_fwd.restype = i
        lib.mla_attn_masked_fwd.argtypes = [p, p, p, p, p, p, p, i, i, i, i, i, f, p, p, sz, p]
        lib.mla_latent_workspace_bytes.restype = sz
        lib.mla_latent_workspace_bytes.argtypes = [i, i, i]
        lib.mla_latent_decode_fwd.restype = i
        lib.mla_latent_decode_fwd.argtypes = [p, p, p, p, p, p, i, i, i, f, p, p, sz, p]
        lib.mla_oproj_workspace_bytes.restype = sz
        lib.mla_oproj_workspace_bytes.argtypes = []
        lib.mla_oproj_fwd.restype = i
        lib.mla_oproj_fwd.argtypes = [p, p, i, i, i, i, p, p, sz, p]
        lib.mla_rope_frequencies.restype = i
        lib.mla_rope_frequencies.argtypes = [ctypes.POINTER(RopeConfig),
                                             ctypes.POINTER(ctypes.c_double),
                                             ctypes.POINTER(ctypes.c_double)]
        lib.mla_rope_table.restype = i
        lib.mla_rope_table.argtypes = [ctypes.POINTER(RopeConfig), i, p, p]
        lib.mla_attn_rope_workspace_bytes.restype = sz
        lib.mla_attn_rope_workspace_bytes.argtypes = [i, i, i, i]
        lib.mla_attn_rope_append_fwd.restype = i
        lib.mla_attn_rope_append_fwd.argtypes = [p, p, p, p, p, p, p, p, p, i, i, i, i, i, f,
                                                 p, i, p, p, sz, p]
        _lib = lib
        return lib


def _status_string(s: int) -> str:
    try:
        return library().mla_status_string(int(s)).decode()
    except Exception:  # pragma: no cover - library missing
        return "libmla_attn.so unavailable"


def mla_attn_workspace_bytes(B: int, H: int, Tq: int, Tk: int) -> int:
    return int(library().mla_attn_workspace_bytes(B, H, Tq, Tk))


def decode_plan(B: int, H: int, Tk: int):
    c, s = ctypes.c_int(), ctypes.c_int()
    rc = library().mla_attn_decode_plan(B, H, Tk, ctypes.byref(c), ctypes.byref(s))
    if rc != 0:
        raise MlaAttnError(rc)
    return c.value, s.value


class Workspace:
    """A zero-initialised device workspace sized for given shapes (grows on demand).

    A workspace serves one stream at a time: calls that may overlap on the GPU (on
    different streams) need workspaces of their own.  The default one, used when a call
    gets none, is shared by every call on its device.
    """

    def __init__(self, device=None):
        self.device = torch.device(device or "cuda")
        self.buf = None

    def get(self, nbytes: int, stream=None) -> torch.Tensor:
        """The buffer, at least nbytes long.  A new buffer is allocated and zero-filled on
        `stream` (the one the call launches on), so the fill precedes the call's kernels."""
        if self.buf is None or self.buf.numel() < nbytes:
            with torch.cuda.stream(stream):
                self.buf = torch.zeros(max(nbytes, 256), dtype=torch.uint8, device=self.device)
        return self.buf


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _check(t, name, dtype, shape, device):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if t.device != device:
        raise ValueError(f"{name} must be on {device}, got {t.device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


class PreparedCall:
    """mla_attn_fwd with its tensors, workspace, stream and options fixed.

    Construction validates everything once; each call re-enqueues the attention core with
    one ctypes call (no per-call Python checks), which matters when the kernels themselves
    take only microseconds.  The tensors are kept alive by this object.
    """

    def __init__(self, q_nope, q_pe, k_nope, k_pe_shared, v, kv_len, past_len: int,
                 softmax_scale: float, out=None, workspace: "Workspace | None" = None,
                 stream=None, path: int = PATH_AUTO, decode_chunk: int = 0):
        lib = library()
        dev = q_nope.device
        if dev.type != "cuda":
            raise ValueError("inputs must be CUDA tensors")
        B, H, Tq = q_nope.shape[:3]
        Tk = k_nope.shape[2]
        bf = torch.bfloat16
        _check(q_nope, "q_nope", bf, (B, H, Tq, 128), dev)
        _check(q_pe, "q_pe", bf, (B, H, Tq, 64), dev)
        _check(k_nope, "k_nope", bf, (B, H, Tk, 128), dev)
        _check(k_pe_shared, "k_pe_shared", bf, (B, Tk, 64), dev)
        _check(v, "v", bf, (B, H, Tk, 128), dev)
        if kv_len is not None:
            _check(kv_len, "kv_len", torch.int32, (B,), dev)
        if out is None:
            out = torch.empty((B, H, Tq, 128), dtype=bf, device=dev)
        _check(out, "out", bf, (B, H, Tq, 128), dev)
        ws_bytes = lib.mla_attn_workspace_bytes(B, H, Tq, Tk)
        if decode_chunk:
            splits = -(-Tk // decode_chunk)
            ws_bytes = max(ws_bytes, 256 + (-(-B * H * splits * 8 // 256)) * 256
                           + B * H * splits * 512)
        s = stream if stream is not None else torch.cuda.current_stream(dev)
        ws = (workspace or _default_workspace(dev)).get(ws_bytes, stream=s)
        self.out = out
        self.device = dev
        self._keep = (q_nope, q_pe, k_nope, k_pe_shared, v, kv_len, out, ws, s)
        self._opts = _Options(int(path), int(decode_chunk))
        self._fn = lib.mla_attn_fwd_ex
        self._args = (_ptr(q_nope), _ptr(q_pe), _ptr(k_nope), _ptr(k_pe_shared), _ptr(v),
                      _ptr(kv_len), B, H, Tq, Tk, int(past_len), float(softmax_scale),
                      _ptr(out), _ptr(ws), ws.numel(), ctypes.c_void_p(s.cuda_stream),
                      ctypes.byref(self._opts))

    def __call__(self):
        if torch.cuda.current_device() != self.device.index:
            with torch.cuda.device(self.device):
                rc = self._fn(*self._args)
        else:
            rc = self._fn(*self._args)
        if rc != 0:
            raise MlaAttnError(rc, "mla_attn_fwd: ")
        return self.out


def mla_attn_fwd(q_nope, q_pe, k_nope, k_pe_shared, v, kv_len, past_len: int,
                 softmax_scale: float, out=None, workspace: Workspace | None = None,
                 stream=None, path: int = PATH_AUTO, decode_chunk: int = 0):
    """out[B,H,Tq,128] (bf16) of the MLA causal-attention core on the current device.

    q_nope [B,H,Tq,128], q_pe [B,H,Tq,64], k_nope [B,H,Tk,128], k_pe_shared [B,Tk,64],
    v [B,H,Tk,128] (bf16, contiguous, CUDA); kv_len [B] int32 on the same device or None.
    Enqueued on ``stream`` (default: torch's current stream); returns ``out``.
    """
    return PreparedCall(q_nope, q_pe, k_nope, k_pe_shared, v, kv_len, past_len,
                        softmax_scale, out, workspace, stream, path, decode_chunk)()


def mla_attn_append_fwd(q_nope, q_pe, k_nope_new, k_pe_new, v_new, k_nope_cache,
                        k_pe_cache, v_cache, kv_len, past_len: int, softmax_scale: float,
                        out=None, workspace: "Workspace | None" = None, stream=None):
    """Append the new key/value rows at [past_len, past_len + Tq) of the caches, then
    attend over rows [0, past_len + Tq).  Caches: k_nope_cache / v_cache [B,H,T_cap,128],
    k_pe_cache [B,T_cap,64]; new rows [B,H,Tq,128] / [B,Tq,64] / [B,H,Tq,128]."""
    lib = library()
    dev = q_nope.device
    if dev.type != "cuda":
        raise ValueError("inputs must be CUDA tensors")
    B, H, Tq = q_nope.shape[:3]
    T_cap = k_nope_cache.shape[2]
    bf = torch.bfloat16
    _check(q_nope, "q_nope", bf, (B, H, Tq, 128), dev)
    _check(q_pe, "q_pe", bf, (B, H, Tq, 64), dev)
    _check(k_nope_new, "k_nope_new", bf, (B, H, Tq, 128), dev)
    _check(k_pe_new, "k_pe_new", bf, (B, Tq, 64), dev)
    _check(v_new, "v_new", bf, (B, H, Tq, 128), dev)
    _check(k_nope_cache, "k_nope_cache", bf, (B, H, T_cap, 128), dev)
    _check(k_pe_cache, "k_pe_cache", bf, (B, T_cap, 64), dev)
    _check(v_cache, "v_cache", bf, (B, H, T_cap, 128), dev)
    if kv_len is not None:
        _check(kv_len, "kv_len", torch.int32, (B,), dev)
    if out is None:
        out = torch.empty((B, H, Tq, 128), dtype=bf, device=dev)
    _check(out, "out", bf, (B, H, Tq, 128), dev)
    s = stream if stream is not None else torch.cuda.current_stream(dev)
    ws = (workspace or _default_workspace(dev)).get(
        lib.mla_attn_workspace_bytes(B, H, Tq, past_len + Tq), stream=s)
    with torch.cuda.device(dev):
        rc = lib.mla_attn_append_fwd(_ptr(q_nope), _ptr(q_pe), _ptr(k_nope_new),
                                     _ptr(k_pe_new), _ptr(v_new), _ptr(k_nope_cache),
                                     _ptr(k_pe_cache), _ptr(v_cache), _ptr(kv_len), B, H, Tq,
                                     T_cap, int(past_len), float(softmax_scale), _ptr(out),
                                     _ptr(ws), ws.numel(), ctypes.c_void_p(s.cuda_stream))
    if rc != 0:
        raise MlaAttnError(rc, "mla_attn_append_fwd: ")
    return out


def mla_attn_masked_fwd(q_nope, q_pe, k_nope, k_pe_shared, v, kv_len, key_mask,
                        past_len: int, softmax_scale: float, out=None,
                        workspace: "Workspace | None" = None, stream=None):
    """Attention with a 2D padding mask on the keys: key_mask [B, Tk] (uint8 or bool CUDA
    tensor, nonzero = attend).  Rows that see no visible key get the mean of all value
    rows (uniform weights)."""
    lib = library()
    dev = q_nope.device
    if dev.type != "cuda":
        raise ValueError("inputs must be CUDA tensors")
    B, H, Tq = q_nope.shape[:3]
    Tk = k_nope.shape[2]
    bf = torch.bfloat16
    _check(q_nope, "q_nope", bf, (B, H, Tq, 128), dev)
    _check(q_pe, "q_pe", bf, (B, H, Tq, 64), dev)
    _check(k_nope, "k_nope", bf, (B, H, Tk, 128), dev)
    _check(k_pe_shared, "k_pe_shared", bf, (B, Tk, 64), dev)
    _check(v, "v", bf, (B, H, Tk, 128), dev)
    if kv_len is not None:
        _check(kv_len, "kv_len", torch.int32, (B,), dev)
    if key_mask.dtype == torch.bool:
        key_mask = key_mask.view(torch.uint8)
    _check(key_mask, "key_mask", torch.uint8, (B, Tk), dev)
    if out is None:
        out = torch.empty((B, H, Tq, 128), dtype=bf, device=dev)
    _check(out, "out", bf, (B, H, Tq, 128), dev)
    s = stream if stream is not None else torch.cuda.current_stream(dev)
    ws = (workspace or _default_workspace(dev)).get(
        lib.mla_attn_masked_workspace_bytes(B, H, Tq, Tk), stream=s)
    with torch.cuda.device(dev):
        rc = lib.mla_attn_masked_fwd(_ptr(q_nope), _ptr(q_pe), _ptr(k_nope), _ptr(k_pe_shared),
                                     _ptr(v), _ptr(kv_len), _ptr(key_mask), B, H, Tq, Tk,
                                     int(past_len), float(softmax_scale), _ptr(out), _ptr(ws),
                                     ws.numel(), ctypes.c_void_p(s.cuda_stream))
    if rc != 0:
        raise MlaAttnError(rc, "mla_attn_masked_fwd: ")
    return out


def mla_latent_decode_fwd(q_nope, q_pe, c_kv, k_pe, w_kvb, kv_len, softmax_scale: float,
                          out=None, workspace: "Workspace | None" = None, stream=None):
    """Decode over the latent cache: q_nope [B,H,128], q_pe [B,H,64], c_kv [B,Tk,512],
    k_pe [B,Tk,64], w_kvb [H*256,512] (kv_b_proj weight), kv_len [B] int32 or None;
    returns out [B,H,128]."""
    lib = library()
    dev = q_nope.device
    if dev.type != "cuda":
        raise ValueError("inputs must be CUDA tensors")
    B, H = q_nope.shape[:2]
    Tk = c_kv.shape[1]
    bf = torch.bfloat16
    _check(q_nope, "q_nope", bf, (B, H, 128), dev)
    _check(q_pe, "q_pe", bf, (B, H, 64), dev)
    _check(c_kv, "c_kv", bf, (B, Tk, 512), dev)
    _check(k_pe, "k_pe", bf, (B, Tk, 64), dev)
    _check(w_kvb, "w_kvb", bf, (H * 256, 512), dev)
    if kv_len is not None:
        _check(kv_len, "kv_len", torch.int32, (B,), dev)
    if out is None:
        out = torch.empty((B, H, 128), dtype=bf, device=dev)
    _check(out, "out", bf, (B, H, 128), dev)
    s = stream if stream is not None else torch.cuda.current_stream(dev)
    ws = (workspace or _default_workspace(dev)).get(lib.mla_latent_workspace_bytes(B, H, Tk),
                                                    stream=s)
    with torch.cuda.device(dev):
        rc = lib.mla_latent_decode_fwd(_ptr(q_nope), _ptr(q_pe), _ptr(c_kv), _ptr(k_pe),
                                       _ptr(w_kvb), _ptr(kv_len), B, H, Tk,
                                       float(softmax_scale), _ptr(out), _ptr(ws), ws.numel(),
                                       ctypes.c_void_p(s.cuda_stream))
    if rc != 0:
        raise MlaAttnError(rc, "mla_latent_decode_fwd: ")
    return out


def mla_oproj_fwd(attn, w_o, out=None, workspace: "Workspace | None" = None, stream=None):
    """Output projection: attn [B,H,T,128], w_o [N, H*128] (bf16, device); returns y [B,T,N]
    with y[b,i] = w_o @ concat_h attn[b,h,i]."""
    lib = library()
    dev = attn.device
    if dev.type != "cuda":
        raise ValueError("inputs must be CUDA tensors")
    B, H, T = attn.shape[:3]
    N = w_o.shape[0]
    bf = torch.bfloat16
    _check(attn, "attn", bf, (B, H, T, 128), dev)
    _check(w_o, "w_o", bf, (N, H * 128), dev)
    if out is None:
        out = torch.empty((B, T, N), dtype=bf, device=dev)
    _check(out, "out", bf, (B, T, N), dev)
    s = stream if stream is not None else torch.cuda.current_stream(dev)
    ws = (workspace or _default_workspace(dev)).get(lib.mla_oproj_workspace_bytes(),
                                                    stream=s)
    with torch.cuda.device(dev):
        rc = lib.mla_oproj_fwd(_ptr(attn), _ptr(w_o), B, H, T, N, _ptr(out), _ptr(ws),
                               ws.numel(), ctypes.c_void_p(s.cuda_stream))
    if rc != 0:
        raise MlaAttnError(rc, "mla_oproj_fwd: ")
    return out


def mla_rope_frequencies(cfg: RopeConfig | None = None):
    """(inv_freq[32] as a list of floats, mscale ratio) computed by the library's host code."""
    cfg = cfg or RopeConfig()
    f = (ctypes.c_double * 32)()
    m = ctypes.c_double()
    rc = library().mla_rope_frequencies(ctypes.byref(cfg), f, ctypes.byref(m))
    if rc != 0:
        raise MlaAttnError(rc, "mla_rope_frequencies: ")
    return list(f), m.value


def mla_rope_table(max_pos: int, cfg: RopeConfig | None = None, device=None, stream=None):
    """Device float32 [max_pos, 64] cos|sin table (times the mscale ratio)."""
    cfg = cfg or RopeConfig()
    dev = torch.device(device or "cuda")
    table = torch.empty((max_pos, 64), dtype=torch.float32, device=dev)
    s = stream if stream is not None else torch.cuda.current_stream(dev)
    with torch.cuda.device(dev):
        rc = library().mla_rope_table(ctypes.byref(cfg), int(max_pos), _ptr(table),
                                      ctypes.c_void_p(s.cuda_stream))
    if rc != 0:
        raise MlaAttnError(rc, "mla_rope_table: ")
    return table


def mla_attn_rope_append_fwd(q_nope, q_pe_raw, k_nope_new, k_pe_new_raw, v_new, k_nope_cache,
                             k_pe_cache, v_cache, kv_len, past_len: int, softmax_scale: float,
                             rope_table, out=None, workspace: "Workspace | None" = None,
                             stream=None):
    """Rotate q_pe_raw / k_pe_new_raw at positions past_len + t (table from mla_rope_table),
    append the new rows (rotated rotary keys) at [past_len, past_len + Tq) of the caches,
    then attend over rows [0, past_len + Tq)."""
    lib = library()
    dev = q_nope.device
    if dev.type != "cuda":
        raise ValueError("inputs must be CUDA tensors")
    B, H, Tq = q_nope.shape[:3]
    T_cap = k_nope_cache.shape[2]
    bf = torch.bfloat16
    _check(q_nope, "q_nope", bf, (B, H, Tq, 128), dev)
    _check(q_pe_raw, "q_pe_raw", bf, (B, H, Tq, 64), dev)
    _check(k_nope_new, "k_nope_new", bf, (B, H, Tq, 128), dev)
    _check(k_pe_new_raw, "k_pe_new_raw", bf, (B, Tq, 64), dev)
    _check(v_new, "v_new", bf, (B, H, Tq, 128), dev)
    _check(k_nope_cache, "k_nope_cache", bf, (B, H, T_cap, 128), dev)
    _check(k_pe_cache, "k_pe_cache", bf, (B, T_cap, 64), dev)
    _check(v_cache, "v_cache", bf, (B, H, T_cap, 128), dev)
    _check(rope_table, "rope_table", torch.float32, (rope_table.shape[0], 64), dev)
    if kv_len is not None:
        _check(kv_len, "kv_len", torch.int32, (B,), dev)
    if out is None:
        out = torch.empty((B, H, Tq, 128), dtype=bf, device=dev)
    _check(out, "out", bf, (B, H, Tq, 128), dev)
    s = stream if stream is not None else torch.cuda.current_stream(dev)
    ws = (workspace or _default_workspace(dev)).get(
        lib.mla_attn_rope_workspace_bytes(B, H, Tq, past_len + Tq), stream=s)
    with torch.cuda.device(dev):
        rc = lib.mla_attn_rope_append_fwd(
            _ptr(q_nope), _ptr(q_pe_raw), _ptr(k_nope_new), _ptr(k_pe_new_raw), _ptr(v_new),
            _ptr(k_nope_cache), _ptr(k_pe_cache), _ptr(v_cache), _ptr(kv_len), B, H, Tq, T_cap,
            int(past_len), float(softmax_scale), _ptr(rope_table), int(rope_table.shape[0]),
            _ptr(out), _ptr(ws), ws.numel(), ctypes.c_void_p(s.cuda_stream))
    if rc != 0:
        raise MlaAttnError(rc, "mla_attn_rope_append_fwd: ")
    return out


def mla_attn_get_status(workspace: Workspace | None = None, device=None, stream=None) -> int:
    """Synchronise and read/clear the device status word (0 = no device-side error)."""
    dev = torch.device(device or "cuda")
    s = stream if stream is not None else torch.cuda.current_stream(dev)
    ws = (workspace or _default_workspace(dev)).get(256, stream=s)
    with torch.cuda.device(dev):
        return int(library().mla_attn_get_status(_ptr(ws), ctypes.c_void_p(s.cuda_stream)))


_default_ws: dict = {}


def _default_workspace(dev) -> Workspace:
    key = str(dev)
    if key not in _default_ws:
        _default_ws[key] = Workspace(dev)
    return _default_ws[key]
