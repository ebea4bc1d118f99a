"""FP64 CPU oracle for ReplaySSM decoding of a Mamba-2 layer.

TEST INFRASTRUCTURE ONLY. Nothing on the product path imports, calls or links this
package: it is used by ``tests/``, by ``__graft_entry__.smoke()`` to check one small
invocation, and by ``bench.py``'s CPU-baseline leg. It shares no code with the CUDA
library; the two meet only in the seeded inputs of :mod:`synthgen`.

Sources: the NVIDIA Developer blog post "ReplaySSM: Rethinking State Storage for Faster
Hybrid-Model Decoding" (sections named in each docstring). Every displayed formula of
that page was lost in extraction; the readings taken are stated where they are used.

Parity pins: every function here is pinned by ``-m "not gpu"`` tests against closed
forms, exact small-integer cases, hand-worked values and format definitions; none is
"parity unpinned".
"""
from . import formats, mamba2  # noqa: F401
