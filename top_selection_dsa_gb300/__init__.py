"""GB300-native DSA lightning-indexer: index logits + masked per-row top-k.

The compute path is the C-ABI library ``libdsa.so`` (hand-written sm_103a CUDA
kernels, declared in ``include/dsa.h``).  ``top_selection_dsa_gb300.api`` is a
thin ctypes binding over it that only marshals torch CUDA tensors into device
pointers and the current stream.  Importing the binding loads the library and
fails loudly when it has not been built: there is no CPU fallback.

``top_selection_dsa_gb300.workloads`` (seeded synthetic inputs) needs no GPU
and no built library, so the package itself loads nothing on import.
"""
from __future__ import annotations

__all__ = [
    "indexer_logits", "topk", "indexer_topk", "indexer_logits_paged",
    "indexer_topk_paged", "workspace_bytes", "DSAError",
]


def __getattr__(name):
    if name in __all__:
        from . import api
        return getattr(api, name)
    raise AttributeError(name)
