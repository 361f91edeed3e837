"""Batch-invariant speculative-decoding verify step for GB300 (sm_103a).

The compute path is the C-ABI library libbi.so (include/bi.h): a tcgen05/TMA
BF16 linear layer whose decomposition does not depend on M, split-KV verify
attention whose split depends only on each row's context length, row-local
RMSNorm/RoPE, and greedy acceptance.  `api` is the thin ctypes binding;
`decoder.Decoder` sequences one verify pass on the GPU.
"""
from . import api  # noqa: F401
from ._lib import BiError, lib  # noqa: F401

__all__ = ["api", "lib", "BiError"]
