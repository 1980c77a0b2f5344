"""GB300-native compute-visible weight-delta sync (PULSESync-style encode/apply).

The compute path is the CUDA library ``libpulse.so`` (C ABI in
``include/pulse.h``); :mod:`.pulse` is its thin Python binding.
"""
from .pulse import (  # noqa: F401
    MX_BLOCK,
    LocoPlan,
    LocoTensorSlot,
    MxPlan,
    MxTensorSlot,
    PackJob,
    Plan,
    PreparedChain,
    PulseError,
    TensorSlot,
    apply,
    compose,
    compose_multi,
    encode,
    encode_noalloc,
    error_string,
    get_error,
    lib,
    library_path,
    loco_accumulate,
    loco_gate,
    mx_apply,
    mx_blocks,
    mx_encode,
    mx_quantize,
    pack_indices,
    unpack_indices,
    tile_elems,
    xor_apply,
    xor_mask,
)
