"""ReplaySSM decoding of a Mamba-2 layer on GB300 (sm_103a).

The compute path is the CUDA library built from ``csrc/`` into ``lib/libreplayssm.so``;
:mod:`.replay` is its thin Python binding (same names as the C ABI in
``include/replayssm.h``). PyTorch supplies device memory and streams only.
"""
from . import replay  # noqa: F401
from .replay import ReplayConfig, ReplayStore  # noqa: F401
