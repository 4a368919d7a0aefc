"""Float64 CPU oracle (test infrastructure only; see exl3_oracle.py)."""
