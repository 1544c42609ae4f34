"""CPU oracle for the Gated DeltaNet forward (test infrastructure only)."""
from .oracle import build, chunked, max_threads, recurrent, recurrent_step

__all__ = ["build", "chunked", "max_threads", "recurrent", "recurrent_step"]
