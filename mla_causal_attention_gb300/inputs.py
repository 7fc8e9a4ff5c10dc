"""Seeded synthetic inputs for the MLA causal-attention core.

This module holds no arithmetic of the attention method: it only draws random tensors of
the shapes the attention core takes.  The same bf16 bit patterns feed both the CUDA
library and the CPU oracle used by the tests.

Recipe.  Every tensor is cut into chunks (one (b, h) slice of a per-head tensor, one b
slice of the shared rotary key); each chunk has its own torch CPU generator seeded from
(seed, tensor id, b, h) by a fixed integer mix, draws float32 N(0,1) values, is multiplied
by the workload's scale factor and is rounded to bf16.  Chunking lets several threads
draw at once and lets a test regenerate one batch row alone.  kv_len comes from its own
generator (integers uniform in [lo, hi], inclusive).
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import torch

from .workloads import Workload

_TENSOR_IDS = {"q_nope": 1, "q_pe": 2, "k_nope": 3, "k_pe_shared": 4, "v": 5, "kv_len": 6,
               "c_kv": 7, "w_kvb": 8, "attn": 9, "w_o": 10}
_MASK64 = (1 << 64) - 1


def chunk_seed(seed: int, tensor: str, b: int, h: int) -> int:
    """A fixed 64-bit mix (splitmix64 finaliser) of the chunk's coordinates."""
    x = (seed * 0x9E3779B97F4A7C15 + _TENSOR_IDS[tensor] * 0xBF58476D1CE4E5B9
         + (b + 1) * 0x94D049BB133111EB + (h + 1) * 0x2545F4914F6CDD1D) & _MASK64
    x ^= x >> 30
    x = (x * 0xBF58476D1CE4E5B9) & _MASK64
    x ^= x >> 27
    x = (x * 0x94D049BB133111EB) & _MASK64
    x ^= x >> 31
    return x & ((1 << 63) - 1)


def _draw(out: torch.Tensor, seed: int, tensor: str, b: int, h: int, factor: float) -> None:
    g = torch.Generator("cpu").manual_seed(chunk_seed(seed, tensor, b, h))
    x = torch.randn(out.shape, generator=g, dtype=torch.float32)
    if factor != 1.0:
        x.mul_(factor)
    out.copy_(x.to(torch.bfloat16))


def draw_kv_len(wl: Workload, seed: int) -> torch.Tensor:
    if wl.kv_len_range is None:
        return torch.full((wl.B,), wl.Tk, dtype=torch.int32)
    lo, hi = wl.kv_len_range
    g = torch.Generator("cpu").manual_seed(chunk_seed(seed, "kv_len", 0, 0))
    return torch.randint(lo, hi + 1, (wl.B,), generator=g, dtype=torch.int64).to(torch.int32)


def make_inputs(wl: Workload, seed: int = 0, pin_memory: bool = False,
                threads: int | None = None, batches=None) -> dict:
    """Host (CPU) bf16 inputs for a workload.

    Returns a dict with q_nope [B,H,Tq,128], q_pe [B,H,Tq,64], k_nope [B,H,Tk,128],
    k_pe_shared [B,Tk,64], v [B,H,Tk,128] (bf16), kv_len [B] (int32), past_len,
    softmax_scale and the workload.  ``batches`` restricts generation to a subset of b
    (the returned tensors then have len(batches) rows, drawn exactly as in the full set).
    """
    kv_len_full = draw_kv_len(wl, seed)
    bs = list(range(wl.B)) if batches is None else [int(b) for b in batches]
    nb = len(bs)
    H, Tq, Tk = wl.H, wl.Tq, wl.Tk
    alloc = dict(dtype=torch.bfloat16, pin_memory=pin_memory)
    t = {
        "q_nope": torch.empty((nb, H, Tq, 128), **alloc),
        "q_pe": torch.empty((nb, H, Tq, 64), **alloc),
        "k_nope": torch.empty((nb, H, Tk, 128), **alloc),
        "k_pe_shared": torch.empty((nb, Tk, 64), **alloc),
        "v": torch.empty((nb, H, Tk, 128), **alloc),
    }
    jobs = []
    for bi, b in enumerate(bs):
        for name in ("q_nope", "q_pe", "k_nope", "v"):
            for h in range(H):
                jobs.append((t[name][bi, h], name, b, h))
        jobs.append((t["k_pe_shared"][bi], "k_pe_shared", b, 0))
    n = threads or min(32, len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity")
                       else (os.cpu_count() or 1))
    f = wl.value_scale
    if n <= 1 or len(jobs) < 4:
        for out, name, b, h in jobs:
            _draw(out, seed, name, b, h, f)
    else:
        with ThreadPoolExecutor(n) as ex:
            list(ex.map(lambda j: _draw(j[0], seed, j[1], j[2], j[3], f), jobs))
    kv_len = kv_len_full[bs].clone()
    if pin_memory:
        kv_len = kv_len.pin_memory()
    t.update(kv_len=kv_len, past_len=wl.past_len, softmax_scale=wl.softmax_scale, workload=wl)
    return t


def make_latent_inputs(wl: Workload, seed: int = 0, pin_memory: bool = False) -> dict:
    """Inputs of decode over the latent cache for a decode workload (Tq = 1): q_nope
    [B,H,128], q_pe [B,H,64], c_kv [B,Tk,512], k_pe [B,Tk,64] ~ N(0,1); the kv_b_proj weight
    w_kvb [H*256,512] ~ N(0, 1/512), so the per-head keys and values it produces from the
    latent rows are ~N(0,1) like the other workloads' inputs (synthetic: no trained
    weights); kv_len drawn as for the workload."""
    B, H, Tk = wl.B, wl.H, wl.Tk
    t = {"q_nope": torch.empty((B, H, 128), dtype=torch.bfloat16),
         "q_pe": torch.empty((B, H, 64), dtype=torch.bfloat16),
         "c_kv": torch.empty((B, Tk, 512), dtype=torch.bfloat16),
         "k_pe": torch.empty((B, Tk, 64), dtype=torch.bfloat16),
         "w_kvb": torch.empty((H * 256, 512), dtype=torch.bfloat16)}
    if pin_memory:
        t = {k: v.pin_memory() for k, v in t.items()}
    jobs = [(t["q_nope"][b], "q_nope", b, 0, 1.0) for b in range(B)]
    jobs += [(t["q_pe"][b], "q_pe", b, 0, 1.0) for b in range(B)]
    jobs += [(t["c_kv"][b], "c_kv", b, 0, 1.0) for b in range(B)]
    jobs += [(t["k_pe"][b], "k_pe_shared", b, 0, 1.0) for b in range(B)]
    jobs += [(t["w_kvb"][h * 256:(h + 1) * 256], "w_kvb", 0, h, 512 ** -0.5) for h in range(H)]
    threads = min(32, os.cpu_count() or 1)
    with ThreadPoolExecutor(threads) as ex:
        list(ex.map(lambda j: _draw(j[0], seed, j[1], j[2], j[3], j[4]), jobs))
    t["kv_len"] = draw_kv_len(wl, seed)
    if pin_memory:
        t["kv_len"] = t["kv_len"].pin_memory()
    return t


def make_oproj_inputs(B: int, H: int, T: int, N: int, seed: int = 0) -> dict:
    """Inputs of the output projection: attn [B,H,T,128] ~ N(0,1) (an attention output's
    shape) and the o_proj weight w_o [N, H*128] ~ N(0, 1/(H*128)), so outputs are ~N(0,1)
    (synthetic: no trained weights)."""
    t = {"attn": torch.empty((B, H, T, 128), dtype=torch.bfloat16),
         "w_o": torch.empty((N, H * 128), dtype=torch.bfloat16)}
    jobs = [(t["attn"][b, h], "attn", b, h, 1.0) for b in range(B) for h in range(H)]
    rows = 256  # weight chunks of 256 output rows
    jobs += [(t["w_o"][r:r + rows], "w_o", 0, r // rows, (H * 128) ** -0.5)
             for r in range(0, N, rows)]
    threads = min(32, os.cpu_count() or 1)
    with ThreadPoolExecutor(threads) as ex:
        list(ex.map(lambda j: _draw(j[0], seed, j[1], j[2], j[3], j[4]), jobs))
    return t
