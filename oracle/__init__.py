"""CPU oracle (test infrastructure only; see llama_oracle.py)."""
