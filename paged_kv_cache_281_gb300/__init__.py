"""Paged-KV attention for GB300 (sm_103a): a C-ABI library and its Python binding.

The hot path — kv_append, paged decode attention (split-K + combine), chunked
causal prefill attention on tcgen05 tensor cores, and block_copy for
copy-on-write — runs in the CUDA kernels of ``libpagedkv.so``; the host block
allocator with refcounts is part of the same library. This package only
builds the library and marshals arguments to it.
"""

from .api import *  # noqa: F401,F403
from .api import __all__  # noqa: F401
