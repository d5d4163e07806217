"""Oracle for the chunkwise gated delta rule forward pass — TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py``
may import this package. It shares no code with the CUDA path and never imports it.

* :func:`kda_recurrence` — the definition: the fp64 token-by-token recurrence, in C
  (``kda_oracle.c``), parallel over (sequence, value head) units.
* :func:`kda_chunked` — the chunkwise restatement of the same result in fp64 numpy
  (``chunked.py``), following the per-chunk steps the pages give, used to pin the chunk
  algebra against the definition.
* :func:`kda_recurrence_bwd` — the backward pass: reverse-mode differentiation of the
  token recurrence in fp64 C (``kda_oracle_bwd.c``).
* :func:`kda_fused_recurrence` — the front-end (q/k L2 norm, beta sigmoid, the Gated
  DeltaNet gate; ``frontend.py``) followed by the recurrence.
"""

from .recurrence import kda_recurrence, oracle_threads  # noqa: F401
from .chunked import kda_chunked, separable_gram, naive_gram  # noqa: F401
from .frontend import kda_fused_recurrence  # noqa: F401
from .backward import kda_recurrence_bwd  # noqa: F401
