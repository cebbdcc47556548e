"""GB300-native fused attention forward + post-attention Ulysses all-to-all.

The product is the C-ABI library ``libattn_a2a.so`` (``include/attn_a2a.h``)
built from ``csrc/`` for sm_103a; ``binding`` exposes the same entry points
to Python. ``workloads`` holds the seeded DiT-shaped input presets and
``burst_gap`` the host-side analysis of the Burst-Gap probe.
"""
from . import workloads  # noqa: F401

__all__ = ["binding", "workloads", "burst_gap", "build"]
