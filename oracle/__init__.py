"""CPU oracle of the draft-sampling / verification path (test infrastructure only)."""
