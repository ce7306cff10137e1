"""GB300 (sm_103a) MXFP4 routed mixture-of-experts expert chain.

The compute path is the C-ABI library libmoe_mxfp4.so (include/moe_mxfp4.h);
this package is its thin binding plus a small layer object that owns device
weights and workspace.
"""

from . import _lib  # noqa: F401  (raises ImportError if the library is not built)
from ._lib import *  # noqa: F401,F403
from .layer import MoeLayer  # noqa: F401
