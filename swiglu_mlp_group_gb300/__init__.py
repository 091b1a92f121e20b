"""GB300 (sm_103a) ConvRot INT8 W8A8 linear and fused SwiGLU MLP (placeholder)."""
