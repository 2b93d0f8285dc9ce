"""fp64 CPU oracle of the GatedDeltaNet layer (test infrastructure only)."""
