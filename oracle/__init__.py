"""fp64 CPU oracle for the MoE FFN layer forward -- test infrastructure only."""
