"""Dilution attention for GB300 (sm_103a): a C-ABI CUDA library and a thin binding.

The compute path lives in ``csrc/`` and is reached through ``libdilution_attn.so``
(see ``include/dilution_attn.h``).  ``binding`` loads it on first use and
raises if it is missing; there is no CPU fallback.
"""
import math

__all__ = ["yarn_tau"]


def yarn_tau(scale: float) -> float:
    """Logit multiplier sqrt(0.1 ln s + 1) for a context extension factor s
    ("YaRN › Attention Temperature Scaling", temperature formula)."""
    return math.sqrt(0.1 * math.log(scale) + 1.0)
