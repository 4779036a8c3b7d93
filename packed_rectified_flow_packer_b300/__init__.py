"""Packed NR-MMDiT block forward with rectified-flow epilogues on one NVIDIA B300 (sm_103a).

The compute lives in libmageflow.so (hand-written CUDA: tcgen05/TMEM/TMA GEMMs with fused
epilogues, a varlen tcgen05 attention kernel, fused LN + modulation prologues, the packer in
C++).  This package is its thin ctypes binding (`binding`) plus device-memory helpers
(`device`).  There is no CPU fallback: importing the binding fails if the library is absent.
"""
from .binding import *  # noqa: F401,F403
from .binding import MageflowError, Plan, lib  # noqa: F401
