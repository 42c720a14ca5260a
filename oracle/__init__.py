"""Float64 CPU oracle (test infrastructure only; see relattn_oracle)."""
