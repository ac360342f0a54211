"""CPU oracle of the Engram layer: test infrastructure only (see engram_oracle)."""
