"""Plain CPU oracle of the routed-expert MoE forward (test infrastructure only)."""
