"""Single-token decode attention over a paged KV cache, for GB300 (sm_103a).

The compute path is libpkv (CUDA kernels behind a C ABI, ``include/pkv.h``);
``paged_kv_cache_273_gb300.pkv`` is its Python binding and
``paged_kv_cache_273_gb300.workloads`` builds seeded synthetic inputs.
Importing the package loads nothing; the binding loads libpkv on first use.
"""
