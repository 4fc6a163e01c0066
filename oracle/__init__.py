"""Double-precision CPU oracle for the block-quantized decode matvec.

Test infrastructure only: the test suite, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference legs of ``bench.py`` may import it; the product path
never does. See ``qmv_oracle`` for the definitions and their sources.
"""
from .qmv_oracle import *  # noqa: F401,F403
from .qmv_oracle import _f64_to_bf16_scalar  # noqa: F401
