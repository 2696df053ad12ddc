"""MiX (Micro-Inverted-Scaling) hot path for one B300: quantisers, A-MiX x W-MX GEMM, K-smoothing."""
