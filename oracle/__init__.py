"""CPU oracle (test infrastructure only): see oracle/mot_oracle.py."""
