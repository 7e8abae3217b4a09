"""Seeded synthetic input generator shared by the oracle side and the CUDA side.

It produces inputs only (weights, activations, gammas, routing biases); it holds none of
the MoE layer's arithmetic."""
