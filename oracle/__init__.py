"""CPU oracle of the DeepSeekMoE FP8 layer (test infrastructure only)."""
