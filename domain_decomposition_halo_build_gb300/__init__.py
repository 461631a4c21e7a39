"""GB300-native eighth-shell domain-decomposition halo exchange.

The compute path is the C-ABI library ``libhalo.so`` (hand-written CUDA for
sm_103a); ``halo`` is its thin ctypes binding.  Import it explicitly:

    from domain_decomposition_halo_build_gb300 import halo
"""
__all__ = ["halo", "synth"]
