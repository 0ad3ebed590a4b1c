"""CPU oracle (test infrastructure only; see w4_oracle.py)."""
