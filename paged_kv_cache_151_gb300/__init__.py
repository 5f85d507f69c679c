"""GB300-native PagedAttention decode: a paged KV-cache write
(``pa_reshape_and_cache``) and decode-step attention over block tables
(``pa_decode``, ``pa_decode_partitioned``), hand-written CUDA for sm_103a
behind a C ABI (``include/pa.h``).

``pa`` is the thin Python binding (argument marshalling only); ``workloads``
builds seeded synthetic inputs.  Importing the package does not load the CUDA
library; the first call does, and fails loudly if it is missing.
"""
__all__ = ["pa", "workloads"]
