"""CPU fp64 oracle for fused online-softmax attention.

TEST INFRASTRUCTURE ONLY. Only the test suite, the smoke check and the bench's
CPU-baseline / reference arm may import this package. The product path (the
CUDA library and its Python binding) never imports, calls or links anything
here, and this package imports nothing from the product.

Pinned by tests/test_oracle_pins.py and tests/test_oracle_rmsnorm_pins.py
(closed forms, invariants, library special cases and brute force on tiny
inputs). Every public function is pinned.
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
from .rmsnorm import (  # noqa: F401
    rms_ref,
    rmsnorm_ref,
    rmsnorm_matmul_ref,
    sumsq_repair,
    sumsq_rolling,
    sumsq_combine,
    l2norm_stable,
)
