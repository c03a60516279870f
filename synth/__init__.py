"""Seeded synthetic inputs shared by the oracle tests and the CUDA path.

This package holds no arithmetic of the decode method itself: it only
describes workload shapes (``presets``), draws seeded random numbers
(``philox``, ``weights``), turns fp32 weight matrices into the block-quantised
storage formats the method consumes (``weights``), and serialises everything
into one flat blob (``blob``).  Both the oracle and the CUDA library read that
blob with readers of their own.
"""

from .presets import PRESETS, ModelSpec, RunSpec, get_preset  # noqa: F401
from .philox import philox4x32_10, uniform_draws  # noqa: F401
from .weights import build_model_blob, prompt_tokens  # noqa: F401
