"""Package for the GB300 DeltaProduct forward path (C-ABI + CUDA kernels)."""
