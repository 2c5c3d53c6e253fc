"""CPU oracle for the fused decode kernels.

TEST INFRASTRUCTURE ONLY. Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline legs of ``bench.py`` may import, call or run anything in this package.
The product path (``memory_bound_decode_fd_gb300``) never imports it and has no
CPU fallback. The oracle shares no code with the CUDA path.
"""

from .fd_oracle import *  # noqa: F401,F403
