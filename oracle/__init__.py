"""Test-only float64 CPU oracle (see lmce_oracle.py).  Not part of the product path."""
