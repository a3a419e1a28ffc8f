"""GB300-native fused-dequantisation GEMV over block-quantised weights.

``synth`` holds the seeded input generators; the CUDA entry points are bound in
``qgemv`` (loaded on first use, and an error if the CUDA library is missing).
"""
