"""fp64 CPU oracle for the ring-attention blockwise forward.

TEST INFRASTRUCTURE: only the tests, the smoke check and the bench's CPU
baseline leg may import anything in this package.  The product path never
does.  It shares no code with the CUDA library.

Parity pins: every function here is pinned by a `-m "not gpu"` test against
something other than itself (a library routine, a closed form, brute force,
or the pages' own worked example).  No function is left unpinned.
"""
from .ref import *  # noqa: F401,F403
