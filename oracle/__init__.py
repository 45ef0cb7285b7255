"""CPU oracle for the Qwen3-style sparse-MoE block forward (test infrastructure).

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library never does, and this
package imports nothing from it.
"""
from .oracle import *  # noqa: F401,F403
