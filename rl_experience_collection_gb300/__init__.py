"""GB300-native fused PPO experience collection.

The compute path is a C-ABI shared library (``include/rollout.h``) built from
``csrc/`` for sm_103a; :mod:`.binding` marshals torch device tensors into it.
Importing the package loads nothing: :mod:`.binding` loads the library on first
use and raises if it is missing.
"""
__all__ = ["workloads", "binding"]
