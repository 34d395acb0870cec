"""Plain, slow fp64 CPU oracle for streaming chunk attention.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import, call or
execute this package: only the tests, the smoke check and the bench's
CPU-baseline / reference arm use it.  It shares no code with the CUDA path
(no kernels, headers, tables or helpers), and it imports nothing from the
``streaming_attention_block_gb300`` package.

Modules
-------
``attention``  masked softmax attention over an explicit token-level chunk
               mask, the streaming (ring) key-set construction, the
               block-causal full-sequence pass and the log-sum-exp merge.
``ring``       a list-based rolling KV cache and the physical slot mapping.
``fp8``        an E4M3 codec written from the OCP 8-bit floating point
               definition, plus the per-(head, chunk) absmax quantiser.

Every function is pinned by ``tests/test_oracle_*.py`` against brute force on
tiny inputs, closed forms, invariants and library special cases.
"""

from . import attention, fp8, ring  # noqa: F401
