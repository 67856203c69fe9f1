"""GB300-native Kimi Delta Attention (KDA) operator.

``kda`` is the Python binding of ``libkda.so`` (C ABI declared in
``include/kda.h``); ``inputs`` draws seeded synthetic problems; ``build``
compiles the library for sm_103a.
"""
from . import inputs  # noqa: F401  (pure torch, no library load)

__all__ = ["kda", "inputs", "build"]
