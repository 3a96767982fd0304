"""GB300-native small-batch MoE expert-FFN decode layer (MXFP8 weights).

The compute path is the C-ABI library libmoedec.so (hand-written sm_103a
CUDA); this package only marshals arguments into it.  Importing the package
is cheap; the first call that needs the library loads it and raises if it has
not been built.
"""
