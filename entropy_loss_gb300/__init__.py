"""Fused linear log-prob / cross-entropy LM head for GB300 (sm_103a).

The compute path is the C-ABI library ``libflp.so`` (hand-written tcgen05 /
TMA / TMEM kernels); ``entropy_loss_gb300.flp`` is its thin ctypes binding.
Importing this package does not load the library; ``flp`` does, and fails
loudly when it is missing.
"""
__all__ = ["flp", "inputs"]
