"""CPU oracle for the block-quantised Linear layer  y = x . dequant(W)^T (+ bias).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference legs of ``bench.py`` may import this package.  The
product path (``bit_weight_quantized_matmul_gb300``) never imports, calls or
links anything here, and this package imports nothing from the product.

The oracle is plain numpy: every quantiser step is one IEEE-754 float32
operation in the order written (numpy applies no FMA contraction to separate
array expressions), and the contraction is an fp64 matrix product.

Modules
-------
formats  scalar formats: E2M1, E4M3, fp16, NF4 codebook
quant    block encoders / decoders: NF4 + double-quant, NVFP4, q4_0, q8_0
linear   the fp64 reference contraction

Parity status: every function here is pinned by ``tests/test_oracle_*.py``
(closed forms, exhaustive code tables, torch casts, brute force, exact rational
arithmetic and hand-worked fixtures under ``tests/golden/``).  The NF4
codebook's digits are pinned to the QLoRA construction and printed table, not
to any bitsandbytes binary (parity with bitsandbytes checkpoints is unpinned).
"""

from . import formats, quant, linear  # noqa: F401
