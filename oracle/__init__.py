"""fp64 CPU oracle of the Stable LatentMoE layer forward (test infrastructure only)."""
