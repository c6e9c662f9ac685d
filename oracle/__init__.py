"""Float64 CPU oracle for block-sparse causal prefill attention.

Test infrastructure only: the tests, the smoke check and the benchmark's
CPU-baseline leg use it; the product path never imports it.  It shares no code
with the CUDA library (``block_sparse_long_fp_gb300``) and does not import it.
"""
from .oracle import *  # noqa: F401,F403
