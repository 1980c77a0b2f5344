"""CPU oracle for the weight-delta encode/apply path.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg use it; the product library never does. The
arithmetic lives in ``pulse_oracle.c`` (plain C, scalar loops, ascending
index order); this module compiles it with gcc and wraps it for numpy arrays.
It imports nothing from the CUDA package.
"""
from .oracle import (  # noqa: F401
    build,
    bf16_rne,
    encode,
    count_changed,
    apply,
    xor_mask,
    xor_apply,
    encode_multi,
    apply_multi,
    xor_mask_multi,
    xor_apply_multi,
)
