"""Block-quantised Linear layers on GB300 (sm_103a): y = x . dequant(W)^T (+ bias).

The compute lives in ``libwq.so`` (hand-written CUDA for sm_103a behind a C ABI,
declared in ``include/wq.h``).  ``wq`` is the thin ctypes binding with the same
names; importing it loads the library and fails loudly when it is missing.
``workloads`` holds the seeded synthetic inputs.
"""
