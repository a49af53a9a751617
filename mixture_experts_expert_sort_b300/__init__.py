"""B300-native MoE expert layer: routing, expert-sort permute, MXFP8 quantise,
tcgen05 grouped GEMMs with fused SwiGLU epilogues, and the unpermute, forward
and backward, behind the C-ABI library ``libmoe``.

The compute library is loaded lazily by :mod:`.binding`; importing the package
itself loads nothing.
"""
__all__ = ["binding", "inputs", "layer"]
