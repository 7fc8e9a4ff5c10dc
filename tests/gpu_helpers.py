"""Shared helpers for the GPU parity tests (device copies, calls, error metrics)."""
import numpy as np
import torch

from oracle import oracle_rows

# Tolerance on bf16 outputs against the exact fp64 oracle (max / mean absolute error).
MAX_ABS_TOL = 2e-2
MEAN_ABS_TOL = 2e-3
KEYS = ("q_nope", "q_pe", "k_nope", "k_pe_shared", "v", "kv_len")


def to_device(inp, device="cuda"):
    d = {k: inp[k].to(device) for k in KEYS}
    d.update(past_len=inp["past_len"], softmax_scale=inp["softmax_scale"])
    return d


def run_gpu(dinp, **kw):
    from mla_causal_attention_gb300 import mla_attn_fwd
    out = mla_attn_fwd(dinp["q_nope"], dinp["q_pe"], dinp["k_nope"], dinp["k_pe_shared"],
                       dinp["v"], dinp["kv_len"], dinp["past_len"], dinp["softmax_scale"], **kw)
    torch.cuda.synchronize()
    return out


def oracle_for(inp, rows=None):
    return oracle_rows(inp["q_nope"], inp["q_pe"], inp["k_nope"], inp["k_pe_shared"],
                       inp["v"], inp["kv_len"], inp["past_len"], inp["softmax_scale"],
                       rows=rows)


def errors(gpu_rows, ref_rows):
    g = gpu_rows.astype(np.float64)
    e = np.abs(g - ref_rows)
    return float(e.max()), float(e.mean())


def assert_close(gpu_rows, ref_rows, label=""):
    mx, mean = errors(gpu_rows, ref_rows)
    print(f"[parity] {label} max|err|={mx:.3e} mean|err|={mean:.3e} n={gpu_rows.shape[0]}")
    assert np.isfinite(gpu_rows).all(), f"{label}: non-finite output"
    assert mx <= MAX_ABS_TOL, f"{label}: max|err| {mx} > {MAX_ABS_TOL}"
    assert mean <= MEAN_ABS_TOL, f"{label}: mean|err| {mean} > {MEAN_ABS_TOL}"


def gpu_rows(out, rows=None):
    o = out.float().cpu().numpy().reshape(-1, 128)
    return o if rows is None else o[np.asarray(rows)]
