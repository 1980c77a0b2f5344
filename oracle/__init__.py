"""CPU oracle for the weight-delta encode/apply path.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg use it; the product library never does. The
arithmetic lives in ``pulse_oracle.c`` (BF16 view), ``mx_oracle.c``
(MXFP8 view), ``mxfp4_oracle.c`` (MXFP4 view), ``nvfp4_oracle.c`` (NVFP4 view), ``compose_oracle.c`` (patch chains), ``loco_oracle.c``
(PULSELoCo gate) and ``pack_oracle.c`` (index packing): plain C, scalar loops, ascending index order; this module
compiles them with gcc and wraps them for numpy arrays. It imports nothing from the CUDA package.
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
    encode_chunked,
    apply_chunked,
    MX_BLOCK,
    e4m3_rne,
    mx_block_scale,
    mx_blocks,
    mxfp8_quantize,
    mxfp8_encode,
    apply_u8,
    mxfp8_apply,
    e2m1_rne,
    mxfp4_block_scale,
    mxfp4_code_bytes,
    mxfp4_quantize,
    mxfp4_encode,
    mxfp4_apply,
    NV_BLOCK,
    nv_blocks,
    nvfp4_tensor_scale,
    nvfp4_quantize,
    nvfp4_encode,
    compose,
    compose_chain,
    loco_gate,
    loco_accumulate,
    PACK_BLOCK,
    PACK_CHUNK,
    pack_indices,
    unpack_indices,
)
