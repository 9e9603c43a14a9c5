"""CPU oracle package (test infrastructure only; see bq_oracle's header)."""
