"""GB300-native mHC layer boundary (n_hc = 4).

The compute path is the C-ABI library ``libmhc.so`` built from ``csrc/`` for
sm_103a; ``ops`` is its thin ctypes binding (argument marshalling only).
"""
