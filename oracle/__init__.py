"""fp64 CPU oracle: test infrastructure only (see ttt_oracle's header)."""
