"""GB300-native (sm_103a) library for the causal-attention core of Kimi K2's MLA.

The compute path is the C-ABI library libmla_attn.so (hand-written CUDA for sm_103a);
``mla_attn_fwd`` marshals torch device tensors into it.  There is no CPU fallback: calls
fail loudly if the library is not built.  The binding is imported on first use so that
the input generator and workload tables can be used without a GPU.
"""
from .workloads import WORKLOADS, Workload  # noqa: F401

_BINDING_NAMES = ("MlaAttnError", "mla_attn_fwd", "mla_attn_workspace_bytes",
                  "mla_attn_get_status", "library", "Workspace", "MlaStatus", "PreparedCall",
                  "mla_attn_append_fwd", "mla_attn_rope_append_fwd", "mla_rope_table",
                  "mla_rope_frequencies", "RopeConfig", "mla_attn_masked_fwd",
                  "mla_latent_decode_fwd", "mla_oproj_fwd")


def __getattr__(name):
    if name in _BINDING_NAMES:
        from . import binding
        return getattr(binding, name)
    raise AttributeError(name)
