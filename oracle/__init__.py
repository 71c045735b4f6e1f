"""CPU oracle for the DSpark verification step (test infrastructure only)."""
