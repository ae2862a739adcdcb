"""fp64 CPU oracle of the DFlash drafter block step (test infrastructure only)."""
