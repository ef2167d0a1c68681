"""A GB300 decode megakernel: an on-GPU interpreter of a static task DAG.

libmk (C ABI, include/mk.h) lowers graph ops to 64-byte task descriptors and
runs one decode step as a persistent sm_103a kernel.  This package is the
Python binding (``_lib``, same names as the C ABI), a graph builder
(``graph.Graph``) and a Llama-style decoder composed on it (``llama``).
"""
from . import _lib  # noqa: F401
from ._lib import MkError  # noqa: F401


def build(force: bool = False, verbose: bool = False) -> str:
    from .build import build as _build
    return _build(force=force, verbose=verbose)
