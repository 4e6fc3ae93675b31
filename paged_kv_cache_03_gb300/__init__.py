"""GB300 (sm_103a) paged attention: exact attention over a paged K/V pool.

The computation lives in libpaged_attn.so (C ABI, include/paged_attn.h);
``binding`` marshals torch tensors into it, ``synth`` draws seeded inputs.
"""
from . import binding, synth  # noqa: F401
from .binding import paged_attention  # noqa: F401
