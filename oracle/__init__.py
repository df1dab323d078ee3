"""CPU oracle for forward attention over a batched, variable-length KV cache.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports, calls or
executes this package: only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` use it.  It shares no code with the CUDA path
(no kernels, headers, tables or helpers); both sides only share the seeded
input generators in ``synth``, which hold none of the method's arithmetic.

Every pinned function is checked in ``tests/test_oracle_*.py`` against things
other than itself: a pure-Python brute force, PyTorch's fp64
``scaled_dot_product_attention``, hand-derived golden values, closed forms and
invariants; ``forward_rows`` (the per-row form the full-size parity tests
use) is checked row by row against ``forward``.
"""
from .reference import (  # noqa: F401
    bf16_to_f64,
    e4m3_decode,
    e4m3_encode,
    fp8_inverse_scale,
    fp8_quantize,
    physical_slots,
    append_kv,
    prepare_prefix,
    gather_sequence,
    visible_mask,
    attend,
    forward,
    forward_rows,
    combine_partials,
    split_forward,
    algorithmic_work,
)
