"""The seeded input generator: deterministic, chunk-addressable, the right shapes/ranges."""
import torch

from mla_causal_attention_gb300.inputs import make_inputs
from mla_causal_attention_gb300.workloads import (WORKLOADS, Workload, algorithmic_bytes,
                                                  algorithmic_flops, softmax_scale_192,
                                                  visible_pairs)


def test_same_seed_same_bits_and_subset_matches():
    wl = Workload("t", 3, 4, 5, 7, 0.5, (3, 12), softmax_scale_192())
    a = make_inputs(wl, seed=3, threads=1)
    b = make_inputs(wl, seed=3, threads=4)
    for k in ("q_nope", "q_pe", "k_nope", "k_pe_shared", "v", "kv_len"):
        assert torch.equal(a[k], b[k]), k
    sub = make_inputs(wl, seed=3, batches=[2])
    for k in ("q_nope", "q_pe", "k_nope", "k_pe_shared", "v", "kv_len"):
        assert torch.equal(sub[k][0], a[k][2]), k
    c = make_inputs(wl, seed=4)
    assert not torch.equal(a["k_nope"], c["k_nope"])


def test_distribution_and_scale():
    wl = WORKLOADS["tiny_prefill"].with_(value_scale=0.5)
    x = make_inputs(wl, seed=0)["k_nope"].float()
    assert abs(x.mean().item()) < 0.02 and abs(x.std().item() - 0.5) < 0.02


def test_workload_sizes():
    w = WORKLOADS
    assert w["long_prefill"].Tk == 4096 and w["chunked_prefill"].Tk == 8192
    assert w["decode_p1000"].Tk == 1001 and w["decode_ragged"].Tk == 8192
    # visible pairs: causal triangle for 4096 tokens, 64 heads
    assert visible_pairs(w["long_prefill"], [4096]) == 64 * 4096 * 4097 // 2
    assert algorithmic_flops(w["long_prefill"], [4096]) == 640 * 64 * 4096 * 4097 // 2
    n = sum(6145 + i for i in range(2048))
    assert visible_pairs(w["chunked_prefill"], [8192] * 4) == 4 * 64 * n
    # decode at cached length 1000: 64 heads x 1001 keys x 512 B + shared key + q + out
    assert algorithmic_bytes(w["decode_p1000"], [1001]) == 32_969_856
