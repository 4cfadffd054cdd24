"""fp64 CPU oracle for the renderer bank-attention path (test infrastructure only).

Only tests, the smoke check and the benchmark's CPU-baseline leg use this
package; the CUDA library never imports it and it imports nothing from the
library.
"""
from .ff_oracle import *  # noqa: F401,F403
