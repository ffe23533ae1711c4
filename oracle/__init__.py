"""CPU oracle of the SonicMoE expert layer: test infrastructure only (see moe_oracle)."""
