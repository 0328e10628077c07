"""fp64 CPU oracle of the TTT inner-loop scan (test infrastructure only)."""
