"""GB300-native 3D Gaussian Splatting training step.

The compute path is libgs.so (hand-written CUDA for sm_103a, C ABI in include/gs.h);
this package holds its ctypes binding (``_native``), the build script (``build``) and
the step orchestrator (``Trainer``).
"""
from . import _native as native
from ._native import GSError, camera, load
from .trainer import Trainer

__all__ = ["native", "GSError", "camera", "load", "Trainer"]
