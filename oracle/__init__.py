"""CPU fp64 oracle (test infrastructure only; see qsa_oracle.py)."""
