"""Seeded synthetic inputs for the tensor-parallel MLP block.

This package holds only shapes, seeds and random draws.  It contains none of
the block's arithmetic, so both the fp64 oracle and the CUDA path can take
their inputs from it without sharing any computation.
"""
from .mlp_inputs import (  # noqa: F401
    MLPShape,
    WORKLOADS,
    workload,
    make_inputs,
    make_ln_grad,
    make_main_grads,
    make_bf16,
    sample_rows,
    sample_ffn_cols,
    reduced_tokens,
    make_saturating_inputs,
    make_zero_block_inputs,
    make_ln_edge_rows,
    LN_EDGE_KINDS,
)
