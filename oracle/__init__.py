"""CPU oracle for the WIDE group-masked projections (test infrastructure only).

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package.  The CUDA library never imports, links or calls
anything here, and nothing here imports the CUDA library.

The arithmetic lives in ``wide_oracle.c`` (plain C, double precision); this
module only builds it with gcc and marshals numpy arrays.  See that file's
header for the passages of "WIDE: Boosting Adaptive LLM Inference via
Token-level Dynamic Width Pruning" each function restates.
"""
from .oracle import (  # noqa: F401
    router,
    attn_decode,
    attn_prefill,
    build,
    library_path,
    reorder,
    proj_mn,
    gate_up,
    proj_k,
    ffn,
    threads,
)
