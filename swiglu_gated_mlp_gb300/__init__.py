"""Fused SwiGLU gated-MLP projection for GB300 (sm_103a): Y = SiLU(A W1) * (A W2)."""
