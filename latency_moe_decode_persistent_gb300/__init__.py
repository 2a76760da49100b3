"""GB300-native persistent megakernel for one speculative-verify decode step of a
mixture-of-experts transformer (single stream, T = k+1 drafted tokens).

The compute path is the C-ABI library ``libmk.so`` built from ``csrc/``; the
Python binding in ``mk.py`` only marshals arguments to it.
"""
