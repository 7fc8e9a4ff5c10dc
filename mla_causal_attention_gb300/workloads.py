"""Named workloads of the MLA causal-attention core (shapes only, no arithmetic).

Head dimensions are those of the Kimi K2 config.json excerpt (page "Kimi K2 · Logits"):
64 attention heads, qk_nope_head_dim 128, qk_rope_head_dim 64, v_head_dim 128, bf16.
The decode shape [B, 64 heads, 1 query, 1001 keys] at cached length 1000 is the tensor
card on the page "Kimi K2 · Similarities".
"""
from __future__ import annotations

import math
from dataclasses import dataclass, replace

import numpy as np

N_HEADS = 64
D_NOPE = 128
D_ROPE = 64
D_V = 128


def softmax_scale_192() -> float:
    """q_head_dim ** -0.5 = 192 ** -0.5, rounded to the float32 the library receives."""
    return float(np.float32(1.0 / math.sqrt(D_NOPE + D_ROPE)))


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    Tq: int
    past_len: int
    value_scale: float = 1.0  # inputs are N(0,1) * value_scale, then bf16
    kv_len_range: tuple | None = None  # (lo, hi) inclusive; None -> every kv_len = Tk
    softmax_scale: float = 0.0

    @property
    def Tk(self) -> int:
        return self.past_len + self.Tq

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


def _wl(name, B, H, Tq, past, vs=1.0, kv=None):
    return Workload(name, B, H, Tq, past, vs, kv, softmax_scale_192())


# The five workloads.  For ragged decode the cache holds Tk = 8192 rows (the top of the
# kv_len range) and past_len = Tk - 1, so causality admits every cached key and kv_len
# alone hides the padding.
WORKLOADS = {
    "tiny_prefill": _wl("tiny_prefill", 1, 64, 16, 0),
    "decode_p1000": _wl("decode_p1000", 1, 64, 1, 1000),
    "decode_ragged": _wl("decode_ragged", 64, 64, 1, 8191, kv=(512, 8192)),
    "long_prefill": _wl("long_prefill", 1, 64, 4096, 0, vs=0.5),
    "chunked_prefill": _wl("chunked_prefill", 4, 64, 2048, 6144),
}


def visible_pairs(wl: Workload, kv_len) -> int:
    """Number of (b, h, i, j) with key j visible to query i (integer count, exact)."""
    kv = np.asarray(kv_len, dtype=np.int64).reshape(-1)
    total = 0
    i = np.arange(wl.Tq, dtype=np.int64)
    for b in range(wl.B):
        lim = np.minimum(i + wl.past_len + 1, kv[b])
        total += int(np.maximum(lim, 0).sum())
    return total * wl.H


def algorithmic_flops(wl: Workload, kv_len) -> int:
    """2 * (192 + 128) FLOP per visible pair: 384 for the scores, 256 for the value mix."""
    return 640 * visible_pairs(wl, kv_len)


def algorithmic_bytes(wl: Workload, kv_len) -> int:
    """Inputs read once plus output written once, bf16.

    Per-head K/V rows count only below kv_len[b] and up to the last key any query of the
    sequence can see; the shared rotary key counts once per (b, key), not once per head.
    """
    kv = np.asarray(kv_len, dtype=np.int64).reshape(-1)
    H, Tq = wl.H, wl.Tq
    total = 0
    for b in range(wl.B):
        keys = int(min(kv[b], wl.past_len + wl.Tq))
        total += keys * (H * (D_NOPE + D_V) + D_ROPE) * 2
        total += H * Tq * (D_NOPE + D_ROPE + D_V) * 2
    return total


# Decode over the latent cache (the 512-wide kv_lora_rank latent rows plus the shared rotary
# key, with the kv_b_proj up-projection absorbed): the two decode workloads above, served
# from a latent cache instead of per-head keys and values.  Synthetic kv_b_proj weights.
LATENT_WORKLOADS = {
    "latent_decode_ragged": WORKLOADS["decode_ragged"],
    "latent_decode_p1000": WORKLOADS["decode_p1000"],
}
D_LAT = 512


def latent_algorithmic_bytes(wl: Workload, kv_len) -> int:
    """Latent rows and rotary keys read once below kv_len (1152 bytes per key), q_nope,
    q_pe and out once per (b, h), and the kv_b_proj weight once (H x 256 x 512 bf16)."""
    kv = np.asarray(kv_len, dtype=np.int64).reshape(-1)
    keys = int(np.minimum(kv, wl.Tk).sum())
    return (keys * (D_LAT + D_ROPE) * 2 + wl.B * wl.H * (D_NOPE + D_ROPE + D_V) * 2
            + wl.H * 256 * D_LAT * 2)
