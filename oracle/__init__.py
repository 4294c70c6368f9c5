"""CPU fp64 oracle (test infrastructure; see attn_sink_oracle)."""
from .attn_sink_oracle import *  # noqa: F401,F403
