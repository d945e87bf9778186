"""Plain, slow fp64 CPU oracle for Block Attention Residuals.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports, calls or
executes anything in this package: only ``tests/``, ``__graft_entry__.smoke()``
and ``bench.py`` (its CPU-baseline leg and its ``--impl reference`` arm) may
use it.  It shares no code with the CUDA path: no kernels, headers, helpers,
tables or pre/post-processing.  Inputs reach it from the seeded generators in
``workloads`` only.

Every function is pinned by ``tests/test_oracle_pins.py`` to facts the pages
and the mathematics fix (worked example, closed forms, invariants, special
cases, an independent high-precision brute force, central differences of the
gradients).  The backward's tolerance scales are pinned by finite
differences of every rounding sensitivity, a closed form at one source, a
float32 evaluation and planted mistakes; the bf16 storage mode of the stack
by a running-state restatement, bit for bit.  No function here is
"parity unpinned"; the one free choice is the final aggregation's
pseudo-query (the pages name the aggregation but not its query), and the
final sources it acts on are pinned independently of that choice.
"""
from .attnres_oracle import (  # noqa: F401
    EPS,
    rms,
    rmsnorm,
    depth_attention,
    depth_attention_lse,
    merge_partial_softmax,
    depth_attention_backward,
    depth_attention_backward_scales,
    backward_rounding_sites,
    backward_scalar_sensitivities,
    block_index,
    position_in_block,
    block_layers,
    num_blocks,
    value_list,
    num_sources,
    round_bf16,
    round_fp32,
    synthetic_layer,
    synthetic_layer_backward,
    block_stack_forward,
    block_stack_backward,
    full_stack_forward,
    StackTrace,
)
