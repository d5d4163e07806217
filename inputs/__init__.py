"""Seeded synthetic inputs shared by the oracle tests, the GPU tests and the benchmark.

This package holds no arithmetic of the method itself: it only draws random numbers,
L2-normalises q and k per token (a data-preparation step), takes log of the sampled
gates, applies sigmoid to the beta logits and rounds to the storage dtype.
"""

from .synth import (WORKLOADS, FrontendInputs, Inputs, Workload, make_frontend_inputs,  # noqa: F401
                    make_inputs, workload_frontend_inputs, workload_inputs)
