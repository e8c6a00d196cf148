"""Oracle package: plain fp64 CPU reference for the multi-head attention
forward pass. Test infrastructure only (see mha_oracle's module docstring)."""

from .mha_oracle import *  # noqa: F401,F403
from .mha_oracle import (BOTTOM, EmptyAllowedRow, MASK_CAUSAL,  # noqa: F401
                         MASK_CAUSAL_PADDING, MASK_NAMES, MASK_NONE,
                         MASK_PADDING)
