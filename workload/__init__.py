"""Seeded synthetic CSR batches of sparse embeddings.

This package only draws inputs. It holds none of the cosine arithmetic, so both
the CPU oracle and the CUDA path can take their inputs from it.
"""
from .generate import (  # noqa: F401
    CONFIGS,
    CsrBatch,
    WorkloadConfig,
    generate_rows,
    generate_side,
    make_pair,
    sample_query_rows,
)
