"""Work accounting of the bench's mask lines, against brute force (CPU)."""
import numpy as np
import pytest

import bench


@pytest.mark.parametrize("Tq,past,pad", [(16, 0, 0), (16, 0, 5), (40, 8, 20), (64, 100, 300),
                                         (130, 0, 129), (7, 3, 10)])
def test_left_padded_visible_pairs_brute_force(Tq, past, pad):
    Tk = past + Tq
    n = sum(1 for i in range(Tq) for j in range(Tk) if j <= i + past and j >= pad)
    assert bench.left_padded_visible_pairs(Tq, past, Tk, pad) == n


def test_left_padded_visible_pairs_long_prefill():
    # 4096 causal rows with the first 512 keys hidden: sum over i >= 512 of (i + 1 - 512).
    assert bench.left_padded_visible_pairs(4096, 0, 4096, 512) == 3584 * 3585 // 2
    assert bench.left_padded_visible_pairs(4096, 0, 4096, 0) == 4096 * 4097 // 2


def test_visible_keys_per_sequence_brute_force():
    rng = np.random.default_rng(7)
    B, Tk = 5, 37
    mask = (rng.random((B, Tk)) > 0.3).astype(np.uint8)
    kv = rng.integers(1, Tk + 1, B)
    want = [sum(1 for j in range(Tk) if mask[b, j] and j < kv[b]) for b in range(B)]
    assert bench.visible_keys_per_sequence(mask, kv).tolist() == want


def test_compact_secondary_entries_stay_short():
    """Thirteen secondary entries of the usual form fit in well under 2 KB of JSON, so the
    whole object survives a 3 KB tail of the output."""
    import json

    res = {"value": 6887.123456, "unit": "GB/s", "ms_per_step": 1.30712345,
           "roofline": {"frac": 1.01481234, "bound": "hbm", "peak": 6786.6,
                        "traffic": 9060000000},
           "clocks": {"sm_mhz": 2070.0, "reasons": []},
           "cpu_baseline": {"value": 30.71234}}
    c = bench.compact(res)
    assert c["v"] == 6887.0 and c["frac"] == 1.01 and c["u"] == "GB/s" and c["cpu"] == 30.7
    sec = {f"workload_name_{k:02d}": c for k in range(13)}
    assert len(json.dumps(sec, separators=(",", ":"))) < 2000
