"""CPU oracle (test infrastructure only; see ess_oracle)."""
