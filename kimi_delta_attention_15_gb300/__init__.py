"""GB300-native (sm_103a) Kimi Delta Attention gated delta rule: chunked
forward and full training backward behind a C ABI (``include/kda.h``).

Importing the package does not load the CUDA library; ``ops`` does, on first
use, and raises if it is missing.
"""
__all__ = ["inputs", "ops"]
