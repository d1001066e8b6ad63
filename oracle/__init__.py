"""CPU oracle of the MoE expert layer (test infrastructure; see moe_ref)."""
