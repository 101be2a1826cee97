"""GB300-native fused KDA (Kimi Delta Attention) single-token decode step and
chunked varlen prefill.

The compute lives in one hand-written CUDA library (``csrc/``) behind a C ABI
(``include/kda_decode.h``); ``kda_decode`` here only marshals torch tensors
into that call.  The library is loaded on first use; a missing library, or
one built for another ABI version, raises instead of falling back to anything
else (``build.build()`` recompiles any source newer than its object).
"""
from .binding import (  # noqa: F401
    KDA_EARLY_PREFETCH,
    KDA_FUSED_GATE,
    KDA_CONV_STATE_SD,
    KDA_OUT_NORM,
    KDA_UPDATE_CONV_STATE,
    KdaDecodeCall,
    MAX_TOKENS_PER_SEQ,
    KdaPrefillCall,
    KdaError,
    kda_chunk_metadata,
    kda_decode,
    kda_prefill,
    kda_status_string,
    library_path,
    load_library,
    longest_first_order,
)
