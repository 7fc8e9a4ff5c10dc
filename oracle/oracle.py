"""ctypes front end of the fp64 CPU oracle (mla_oracle.c).

TEST INFRASTRUCTURE ONLY.  Nothing in the product package imports this module.

The oracle takes the same bf16 bit patterns the CUDA library takes (as numpy uint16
arrays or CPU torch bfloat16 tensors) and returns exact fp64 output rows of the attention
core described on the page "Kimi K2 · Similarities" (section "Contextual evidence from
Query-key similarity"): scores over the concatenated 192-wide query/key, scale, additive
causal/padding mask, softmax, weighted sum of the 128-wide values.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mla_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD, "libmla_oracle.so")
_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return _LIB


def build_oracle(force: bool = False) -> str:
    """Compile mla_oracle.c with gcc (IEEE arithmetic: no fast-math, no FMA contraction)."""
    os.makedirs(_BUILD, exist_ok=True)
    stale = (not os.path.exists(_LIB)) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC)
    if force or stale:
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
               "-pthread", "-Wall", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            # MLA_ORACLE_LIB points the loader at another build of mla_oracle.c; the
            # mutation test uses it to check that the pins fail on planted mistakes.
            path = os.environ.get("MLA_ORACLE_LIB")
            if not path:
                path = build_oracle()
            lib = ctypes.CDLL(path)
            p = ctypes.c_void_p
            i64 = ctypes.c_int64
            lib.mla_oracle_rows.restype = ctypes.c_int
            lib.mla_oracle_rows.argtypes = [p, p, p, p, p, p, i64, i64, i64, i64, i64,
                                            ctypes.c_float, p, i64, ctypes.c_int, ctypes.c_int,
                                            p, p]
            lib.mla_oracle_rows_mask.restype = ctypes.c_int
            lib.mla_oracle_rows_mask.argtypes = [p, p, p, p, p, p, p, i64, i64, i64, i64, i64,
                                                 ctypes.c_float, p, i64, ctypes.c_int,
                                                 ctypes.c_int, p, p]
            lib.mla_oracle_latent_rows.restype = ctypes.c_int
            lib.mla_oracle_latent_rows.argtypes = [p, p, p, p, p, p, i64, i64, i64, i64, i64,
                                                   ctypes.c_float, p, i64, ctypes.c_int, p]
            lib.mla_oracle_round_bf16.restype = ctypes.c_double
            lib.mla_oracle_round_bf16.argtypes = [ctypes.c_double]
            lib.mla_oracle_rows_rope.restype = ctypes.c_int
            lib.mla_oracle_rows_rope.argtypes = [p, p, p, p, p, p, i64, i64, i64, i64, i64,
                                                 ctypes.c_float, p, i64, ctypes.c_int, p, p,
                                                 ctypes.c_double]
            d = ctypes.c_double
            lib.mla_oracle_yarn.restype = None
            lib.mla_oracle_yarn.argtypes = [d, d, d, d, d, d, d, p, p]
            lib.mla_oracle_rotate.restype = ctypes.c_int
            lib.mla_oracle_rotate.argtypes = [p, p, i64, p, d, p]
            lib.mla_oracle_oproj_rows.restype = ctypes.c_int
            lib.mla_oracle_oproj_rows.argtypes = [p, p, i64, i64, i64, i64, p, i64,
                                                  ctypes.c_int, p]
            _lib = lib
    return _lib


def _bits(x) -> np.ndarray:
    """bf16 bit patterns as a C-contiguous uint16 numpy array (no copy where possible)."""
    if isinstance(x, np.ndarray):
        assert x.dtype == np.uint16
        return np.ascontiguousarray(x)
    import torch  # local: only tensors need it

    assert x.dtype == torch.bfloat16 and x.device.type == "cpu"
    return np.ascontiguousarray(x.contiguous().view(torch.int16).numpy().view(np.uint16))


def _threads(n):
    if n:
        return int(n)
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def oracle_rows(q_nope, q_pe, k_nope, k_pe_shared, v, kv_len, past_len: int,
                softmax_scale: float, rows=None, mode: str = "exact", threads: int | None = None,
                return_wsum: bool = False, key_mask=None):
    """Exact fp64 output rows.

    Shapes: q_nope [B,H,Tq,128], q_pe [B,H,Tq,64], k_nope [B,H,Tk,128],
    k_pe_shared [B,Tk,64], v [B,H,Tk,128] (bf16), kv_len [B] int32 or None,
    key_mask [B,Tk] (nonzero = key visible) or None.
    rows: flat indices (b*H + h)*Tq + i, or None for all rows in that order.
    Returns float64 [n_rows,128] (and the per-row weight sum if asked).
    """
    lib = _load()
    qn, qr, kn, kr, vv = (_bits(t) for t in (q_nope, q_pe, k_nope, k_pe_shared, v))
    B, H, Tq, dn = qn.shape
    Tk = kn.shape[2]
    assert dn == 128 and qr.shape == (B, H, Tq, 64) and kn.shape == (B, H, Tk, 128)
    assert kr.shape == (B, Tk, 64) and vv.shape == (B, H, Tk, 128)
    kvl = None
    if kv_len is not None:
        kvl = np.ascontiguousarray(np.asarray(kv_len, dtype=np.int32).reshape(B))
    if rows is None:
        n = B * H * Tq
        rows_arr = None
    else:
        rows_arr = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1))
        n = rows_arr.size
    out = np.empty((n, 128), dtype=np.float64)
    wsum = np.empty((n,), dtype=np.float64)
    m = {"exact": 0, "eager": 1}[mode]
    ptr = lambda a: None if a is None else a.ctypes.data  # noqa: E731
    if key_mask is None:
        rc = lib.mla_oracle_rows(ptr(qn), ptr(qr), ptr(kn), ptr(kr), ptr(vv), ptr(kvl),
                                 B, H, Tq, Tk, int(past_len), float(softmax_scale),
                                 ptr(rows_arr), n, m, _threads(threads), ptr(out), ptr(wsum))
    else:
        if hasattr(key_mask, "numpy"):
            key_mask = key_mask.cpu().numpy()
        km = np.ascontiguousarray((np.asarray(key_mask) != 0).astype(np.uint8).reshape(B, Tk))
        rc = lib.mla_oracle_rows_mask(ptr(qn), ptr(qr), ptr(kn), ptr(kr), ptr(vv), ptr(kvl),
                                      ptr(km), B, H, Tq, Tk, int(past_len),
                                      float(softmax_scale), ptr(rows_arr), n, m,
                                      _threads(threads), ptr(out), ptr(wsum))
    if rc != 0:
        raise ValueError(f"oracle rejected its arguments (code {rc})")
    return (out, wsum) if return_wsum else out


def oracle_full(inp: dict, mode: str = "exact", threads: int | None = None) -> np.ndarray:
    """All output rows for an input dict from the seeded generator, shaped [B,H,Tq,128]."""
    B, H, Tq = inp["q_nope"].shape[:3]
    o = oracle_rows(inp["q_nope"], inp["q_pe"], inp["k_nope"], inp["k_pe_shared"], inp["v"],
                    inp["kv_len"], inp["past_len"], inp["softmax_scale"], mode=mode,
                    threads=threads)
    return o.reshape(B, H, Tq, 128)


def round_bf16(x: float) -> float:
    """The eager-emulation diagnostic's round-to-bf16 (exposed so a test can pin it)."""
    return _load().mla_oracle_round_bf16(float(x))


def yarn(theta: float, factor: float, orig_max_pos: int, beta_fast: float, beta_slow: float,
         mscale: float, mscale_all_dim: float):
    """The 32 YaRN rotary frequencies and the mscale ratio on cos/sin (fp64)."""
    lib = _load()
    f = np.zeros(32, dtype=np.float64)
    r = np.zeros(1, dtype=np.float64)
    lib.mla_oracle_yarn(float(theta), float(factor), float(orig_max_pos), float(beta_fast),
                        float(beta_slow), float(mscale), float(mscale_all_dim), f.ctypes.data,
                        r.ctypes.data)
    return f, float(r[0])


def oracle_latent_rows(q_nope, q_pe, c_kv, k_pe, w_kvb, kv_len, past_len: int,
                       softmax_scale: float, rows=None, threads: int | None = None):
    """Output rows of attention over the latent cache, non-absorbed form, fp64.

    q_nope [B,H,Tq,128], q_pe [B,H,Tq,64], c_kv [B,Tk,512], k_pe [B,Tk,64] (bf16),
    w_kvb [H*256,512] (bf16, kv_b_proj weight), kv_len [B] or None.  Returns [n_rows,128].
    """
    lib = _load()
    qn, qr, c, kr, w = (_bits(t) for t in (q_nope, q_pe, c_kv, k_pe, w_kvb))
    B, H, Tq, _ = qn.shape
    Tk = c.shape[1]
    assert c.shape == (B, Tk, 512) and kr.shape == (B, Tk, 64) and w.shape == (H * 256, 512)
    kvl = None if kv_len is None else np.ascontiguousarray(
        np.asarray(kv_len, dtype=np.int32).reshape(B))
    rows_arr = None if rows is None else np.ascontiguousarray(
        np.asarray(rows, dtype=np.int64).reshape(-1))
    n = B * H * Tq if rows is None else rows_arr.size
    out = np.empty((n, 128), dtype=np.float64)
    ptr = lambda a: None if a is None else a.ctypes.data  # noqa: E731
    rc = lib.mla_oracle_latent_rows(ptr(qn), ptr(qr), ptr(c), ptr(kr), ptr(w), ptr(kvl), B, H,
                                    Tq, Tk, int(past_len), float(softmax_scale), ptr(rows_arr),
                                    n, _threads(threads), ptr(out))
    if rc != 0:
        raise ValueError(f"oracle rejected its arguments (code {rc})")
    return out


def rotate(x, positions, inv_freq, mscale: float):
    """The rotary step alone: rows of x ([..., 64] bf16) rotated at positions (broadcast to
    x's leading shape, one per row); returns fp64 [..., 64]."""
    lib = _load()
    xb = _bits(x)
    shape = xb.shape
    assert shape[-1] == 64
    rows = np.ascontiguousarray(xb.reshape(-1, 64))
    pos = np.ascontiguousarray(np.broadcast_to(np.asarray(positions, dtype=np.int64),
                                               shape[:-1]).reshape(-1))
    out = np.empty((rows.shape[0], 64), dtype=np.float64)
    f = np.ascontiguousarray(np.asarray(inv_freq, dtype=np.float64).reshape(32))
    rc = lib.mla_oracle_rotate(rows.ctypes.data, pos.ctypes.data, rows.shape[0], f.ctypes.data,
                               float(mscale), out.ctypes.data)
    if rc != 0:
        raise ValueError(f"oracle rejected its arguments (code {rc})")
    return out.reshape(shape)


def oracle_rows_rope(q_nope, q_pe_raw, k_nope, k_pe, v, kv_len, past_len: int,
                     softmax_scale: float, inv_freq, mscale: float, rows=None,
                     threads: int | None = None):
    """Like oracle_rows, with the rotary step first: q_pe_raw unrotated (query i at position
    past_len + i); k_pe rows j >= past_len unrotated new keys (position j); rows below
    past_len are cached keys, already rotated."""
    lib = _load()
    qn, qr, kn, kr, vv = (_bits(t) for t in (q_nope, q_pe_raw, k_nope, k_pe, v))
    B, H, Tq, _ = qn.shape
    Tk = kn.shape[2]
    kvl = None if kv_len is None else np.ascontiguousarray(
        np.asarray(kv_len, dtype=np.int32).reshape(B))
    rows_arr = None if rows is None else np.ascontiguousarray(
        np.asarray(rows, dtype=np.int64).reshape(-1))
    n = B * H * Tq if rows is None else rows_arr.size
    out = np.empty((n, 128), dtype=np.float64)
    f = np.ascontiguousarray(np.asarray(inv_freq, dtype=np.float64).reshape(32))
    ptr = lambda a: None if a is None else a.ctypes.data  # noqa: E731
    rc = lib.mla_oracle_rows_rope(ptr(qn), ptr(qr), ptr(kn), ptr(kr), ptr(vv), ptr(kvl), B, H,
                                  Tq, Tk, int(past_len), float(softmax_scale), ptr(rows_arr), n,
                                  _threads(threads), ptr(out), ptr(f), float(mscale))
    if rc != 0:
        raise ValueError(f"oracle rejected its arguments (code {rc})")
    return out


def oracle_oproj_rows(attn, w, rows=None, threads: int | None = None):
    """Output projection (o_proj) of attention output rows, fp64.

    attn [B,H,T,128] bf16 (the attention core's output), w [N, H*128] bf16 (nn.Linear
    weight, out_features x in_features).  Row r is (b, i) = divmod(rows[r], T), its input
    the heads' outputs concatenated in head order.  Returns [n_rows, N].
    """
    lib = _load()
    a, wb = _bits(attn), _bits(w)
    B, H, T, dv = a.shape
    N, K = wb.shape
    assert dv == 128 and K == H * 128
    if rows is None:
        rows_arr, n_rows, rows_p = None, B * T, None
    else:
        rows_arr = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        n_rows, rows_p = rows_arr.size, rows_arr.ctypes.data_as(ctypes.c_void_p)
    out = np.empty((n_rows, N), dtype=np.float64)
    rc = lib.mla_oracle_oproj_rows(a.ctypes.data_as(ctypes.c_void_p),
                                   wb.ctypes.data_as(ctypes.c_void_p), B, H, T, N, rows_p,
                                   n_rows, _threads(threads),
                                   out.ctypes.data_as(ctypes.c_void_p))
    if rc != 0:
        raise ValueError(f"mla_oracle_oproj_rows failed with code {rc}")
    return out
