"""CPU oracle for the weight-absorbed MLA path (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. The library under
``mla_latent_kv_11_gb300/`` never does, and shares no code with it.
"""
from .mla_oracle import *  # noqa: F401,F403
from . import mla_oracle  # noqa: F401
