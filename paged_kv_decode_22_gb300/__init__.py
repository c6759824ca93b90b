"""GB300 (sm_103a) paged-KV decode attention and KV-cache copy kernels.

The compute lives in the CUDA library ``libpkd.so`` (C ABI: include/pkd.h);
``paged_kv_decode_22_gb300.ops`` re-exports its thin Python binding.  Build
the library with ``paged_kv_decode_22_gb300.build.build()``.
"""
