"""GB300-native KroQuant MXFP4 activation quantizer.

The compute path is the C-ABI shared library built from ``csrc/`` for
sm_103a; ``kq`` is its thin ctypes binding (argument marshalling only) and
``synth`` the seeded synthetic-input generator.  Importing the package loads
nothing; the library is loaded on first use of ``kq`` and a missing library
raises instead of falling back to anything else.
"""
__all__ = ["kq", "synth"]
