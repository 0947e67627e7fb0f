"""fp64 CPU oracle for exact attention: TEST INFRASTRUCTURE ONLY.

Used by the tests, the smoke check and the benchmark's CPU-baseline leg; never by
the CUDA library or its Python binding, with which it shares no code.
"""
