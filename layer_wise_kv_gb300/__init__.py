"""Layer-wise KV-cache sparsification over a paged KV cache, on one GB300.

The compute lives in ``libkvs.so`` (hand-written CUDA for sm_103a behind the C
ABI in ``include/kvs.h``); :mod:`layer_wise_kv_gb300.kvs` is its binding and
:mod:`layer_wise_kv_gb300.pipeline` strings the calls together into the
prefill+sparsify and decode steps.
"""
from . import kvs  # noqa: F401
