"""fp64 CPU oracle of the Kimi K2 MLA causal-attention core.

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the CPU-baseline leg of the
benchmark use it to check and time the CUDA library.  The library never imports it.
"""
from .oracle import (build_oracle, oracle_rows, oracle_full, oracle_rows_rope,  # noqa: F401
                     round_bf16, library_path, rotate, yarn,
                     oracle_latent_rows, oracle_oproj_rows)
