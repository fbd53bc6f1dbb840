"""CPU fp64 oracle for fused online-softmax attention.

TEST INFRASTRUCTURE ONLY. Only the test suite, the smoke check and the bench's
CPU-baseline / reference arm may import this package. The product path (the
CUDA library and its Python binding) never imports, calls or links anything
here, and this package imports nothing from the product.

Pinned by tests/test_oracle_pins.py (closed forms, invariants, a library
special case and brute force on tiny inputs). Every public function is pinned.
"""
from .attention import (  # noqa: F401
    attend_head,
    attention_ref,
    attention_backward_ref,
    decode_ref,
    decode_split_partials_ref,
    combine_ref,
    online_softmax_rolling,
    naive_fused_exp_sum,
    repair,
)
