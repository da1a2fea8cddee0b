"""GB300 (sm_103a) low-bit KV-cache quantization with fused-dequant decode attention.

The compute path is the C-ABI library ``libkvq.so`` (hand-written CUDA, see
``include/kvq.h``); ``kvq`` is its thin Python binding.  ``synthetic`` draws the
seeded workloads used by the tests and the benchmark.
"""
__version__ = "0.1.0"
