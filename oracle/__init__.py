"""CPU oracle package (test infrastructure only; see h3q_oracle's docstring)."""
