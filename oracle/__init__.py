"""fp64 CPU oracle of the Gated DeltaNet token mixer (test infrastructure only).

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package; the CUDA library never does.
"""

from .gdn_oracle import (  # noqa: F401
    CHUNK, CONV_K, causal_conv1d, chunk_gated_delta_rule, conv_gating, decode_step,
    gated_rmsnorm, gating, l2norm, mixer_prefill, recurrent_gated_delta_rule, sigmoid,
    silu, softplus,
)
