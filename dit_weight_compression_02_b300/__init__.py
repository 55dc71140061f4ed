"""EntroPack for B300: entropy-coded E8 weight streams decoded by sm_103a kernels.

See include/entropack.h for the C ABI and the stream format (version 1).
"""
from .api import *  # noqa: F401,F403
from .api import __all__  # noqa: F401
