"""Decode over the latent cache (mla_latent_decode_fwd) against the oracle's non-absorbed
rows: the per-head no-rope keys and values the kv_b_proj weight would produce from the
latent rows, then the usual attention."""
import numpy as np
import pytest
import torch

from mla_causal_attention_gb300 import binding
from mla_causal_attention_gb300.workloads import softmax_scale_192
from gpu_helpers import assert_close
from oracle import oracle_latent_rows

pytestmark = pytest.mark.gpu


def _case(B, H, Tk, kv=None, seed=0):
    g = torch.Generator("cpu").manual_seed(seed)
    mk = lambda *s: torch.randn(*s, generator=g).to(torch.bfloat16)  # noqa: E731
    d = dict(q_nope=mk(B, H, 128), q_pe=mk(B, H, 64), c_kv=mk(B, Tk, 512), k_pe=mk(B, Tk, 64),
             w_kvb=(torch.randn(H * 256, 512, generator=g) / 512 ** 0.5).to(torch.bfloat16),
             kv_len=None)
    if kv is not None:
        d["kv_len"] = torch.randint(kv[0], kv[1] + 1, (B,), generator=g, dtype=torch.int32)
    return d


def _gpu(d):
    c = {k: (None if v is None else v.cuda()) for k, v in d.items()}
    out = binding.mla_latent_decode_fwd(c["q_nope"], c["q_pe"], c["c_kv"], c["k_pe"],
                                        c["w_kvb"], c["kv_len"], softmax_scale_192())
    torch.cuda.synchronize()
    assert binding.mla_attn_get_status(device=out.device) == 0
    return out.float().cpu().numpy().reshape(-1, 128)


def _oracle(d, rows=None):
    Tk = d["c_kv"].shape[1]
    return oracle_latent_rows(d["q_nope"][:, :, None], d["q_pe"][:, :, None], d["c_kv"],
                              d["k_pe"], d["w_kvb"], d["kv_len"], Tk - 1, softmax_scale_192(),
                              rows=rows)


@pytest.mark.parametrize("B,H,Tk,kv", [
    (1, 64, 1, None),          # a single key
    (2, 64, 128, None),        # exactly one tile
    (2, 64, 300, None),        # a ragged last tile
    (3, 64, 1001, (1, 1001)),  # ragged kv_len, several splits
    (1, 64, 1001, None),       # the decode shape at cached length 1000
    (2, 16, 700, (200, 700)),  # fewer heads than the MMA's 64 columns
    (5, 64, 2000, (1, 2000)),  # one split per sequence on a busy GPU
    (70, 8, 200, (1, 200)),    # more sequences than one projection block (64) holds
    (1, 8, 8192, None),        # 64 tiles over 64 CTAs: the combine's weights in two rounds
    (300, 4, 128, (1, 128)),   # more sequences than CTAs: each CTA walks several
])
def test_latent_matches_oracle(B, H, Tk, kv):
    d = _case(B, H, Tk, kv, seed=B * 100 + Tk)
    assert_close(_gpu(d), _oracle(d), f"latent B{B} H{H} Tk{Tk}")


def test_latent_ragged_batch_sampled():
    d = _case(16, 64, 8192, (512, 8192), seed=7)
    got = _gpu(d)
    rows = [b * 64 + h for b in range(16) for h in (0, 31, 63)]
    assert_close(got[rows], _oracle(d, rows), "latent B16 Tk8192 sampled")


def test_latent_decode_ragged_full_size_sampled():
    """The bench's latent workload (64 sequences x 64 heads, kv_len ~ U[512, 8192], its
    generator and launch plan): twelve rows against the oracle."""
    from mla_causal_attention_gb300.inputs import make_latent_inputs
    from mla_causal_attention_gb300.workloads import LATENT_WORKLOADS
    w = LATENT_WORKLOADS["latent_decode_ragged"]
    d = make_latent_inputs(w, seed=0)
    got = _gpu(d)
    kv = d["kv_len"].numpy()
    bs = sorted({int(np.argmin(kv)), int(np.argmax(kv)), 0, w.B - 1})
    rows = [b * w.H + h for b in bs for h in (0, 31, w.H - 1)]
    assert_close(got[rows], _oracle(d, rows), "latent_decode_ragged full, sampled")
