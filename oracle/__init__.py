"""CPU oracle for the Gated DeltaNet forward (test infrastructure only)."""
from .oracle import (build, causal_conv1d_silu, chunked, decode_gates, gated_rmsnorm, l2_normalise, max_threads,
                     num_procs, recurrent, recurrent_step, recurrent_step_gated, round_to_bf16, set_threads, silu,
                     softplus)

__all__ = ["build", "causal_conv1d_silu", "chunked", "decode_gates", "gated_rmsnorm", "l2_normalise", "max_threads",
           "num_procs", "recurrent", "recurrent_step", "recurrent_step_gated", "round_to_bf16", "set_threads", "silu",
           "softplus"]
