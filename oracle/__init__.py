"""fp64 CPU oracle of the fused KDA decode step, its multi-token (speculative)
form and the varlen prefill.

TEST INFRASTRUCTURE ONLY: the test-suite, the smoke check and the benchmark's
CPU-baseline leg load it; the product library never does, and the two share
no code.  The formulation it computes is written out in ``kda_oracle.h``.
"""
from .kda_oracle import (  # noqa: F401
    OracleResult,
    build,
    decode,
    decode_multi,
    prefill,
    lib,
    round_bf16,
    bf16_to_f64,
    causal_conv,
    silu,
    sigmoid,
    l2norm,
    gated_delta_update,
    readout,
    gated_rmsnorm,
    softplus,
    kda_gate,
)
