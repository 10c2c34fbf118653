"""GB300 (sm_103a) tensor-parallel transformer MLP block: a C-ABI CUDA library
(libmlpb) and its thin ctypes binding."""
from .mlpb import *  # noqa: F401,F403
from .mlpb import MLPBlock, MLPBError, MLPBranch, load_library  # noqa: F401
