"""fq: Qwen3 quantized single-token decode on GB300 (sm_103a).

The decode step runs in the CUDA library ``libfq.so`` behind the C ABI of
``include/fq.h``; :mod:`.fq` is its ctypes binding and :mod:`.build` compiles it.
"""
from . import fq  # noqa: F401
from .fq import FqError  # noqa: F401
