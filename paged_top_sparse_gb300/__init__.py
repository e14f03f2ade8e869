"""paged_top_sparse_gb300: paged block-sparse prefill attention on GB300 (sm_103a).

The compute lives in a C-ABI shared library (``include/sparse_prefill.h``) built from the
CUDA sources under ``csrc/``; ``binding`` is its thin ctypes front end.  Import
``paged_top_sparse_gb300.binding`` for the calls; this package module stays light so that
``synth`` (input generation) can be imported without the library.
"""
