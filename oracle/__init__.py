"""CPU fp64 oracle (test infrastructure only; see moe_oracle.py)."""
