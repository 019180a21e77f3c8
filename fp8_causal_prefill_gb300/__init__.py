"""GB300-native causal FP8 / BF16 prefill attention with the ZYFA numerics (Lean P, per-64-key
power-of-two block scaling, rounded-row-sum normalisation)."""
