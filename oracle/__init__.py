"""CPU reference implementation of the KroQuant MXFP4 activation quantizer.

TEST INFRASTRUCTURE ONLY: imported by the tests, the smoke check and the
CPU-baseline leg of the benchmark, never by the product path.
"""
