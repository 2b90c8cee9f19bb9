"""libpagedattn: decode attention over a paged KV cache, hand-written for GB300 (sm_103a).

The compute lives in ``csrc/`` behind a C ABI (``include/pagedattn.h``);
``binding`` marshals torch tensors into those calls.  Importing this package
does not load the shared library; the first call does, and it raises if the
library was not built (there is no CPU fallback).
"""

__all__ = ["binding", "workloads", "accounting", "build"]
