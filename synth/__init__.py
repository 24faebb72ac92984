"""Seeded synthetic inputs and workload shapes (no method arithmetic)."""
from .configs import (C1_TINY, C2_MID, C3_14B, C4_CONVKV, C5_FP8, CONFIGS,  # noqa: F401
                      PoseRecipe, StreamConfig)
from . import gen  # noqa: F401
