"""CPU oracle (test infrastructure only; see tdp_oracle's header)."""
