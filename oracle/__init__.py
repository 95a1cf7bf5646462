"""CPU oracle for MoE dispatch/combine -- test infrastructure only (see ref.py)."""
