"""GB300 (sm_103a) implementation of the DSpark Markov-head drafting hot path.

The compute lives in ``csrc/`` (hand-written CUDA kernels behind the C ABI of
``include/dspark.h``); ``binding`` is the thin ctypes layer over it and
``build`` compiles the library in-tree.
"""

from . import build  # noqa: F401
from .binding import (  # noqa: F401
    Confidence, Context, DSparkError, confidence, gate, markov_draft, markov_logits,
    selector_scores, selector_walk,
)

__all__ = ["Confidence", "Context", "DSparkError", "confidence", "gate", "markov_draft",
           "markov_logits", "selector_scores", "selector_walk", "build"]
