"""CPU oracle for the MXFP4 routed-MoE expert chain. Test infrastructure only.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. The library under
``mxfp4_mixture_experts_bucket_gb300`` never does, and shares no code with it.
"""

from . import moe_oracle, brute  # noqa: F401
