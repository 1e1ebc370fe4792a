"""Budgeted KV-cache compression (probe scoring, global Add/Split auction,
RoPE-consistent prototype merging, ragged packing) and ragged GQA decode for
one GB300.  The compute lives in libkvc.so (hand-written CUDA for sm_103a);
``kvc`` is its ctypes binding and ``pipeline`` a helper that owns device
buffers and workspaces."""
from . import kvc  # noqa: F401
