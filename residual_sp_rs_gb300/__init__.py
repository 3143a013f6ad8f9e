"""GB300-native (sm_103a) sequence-parallel region hot path.

The compute lives in ``libspfuse.so`` (C ABI, hand-written CUDA kernels);
this package only marshals arguments to it.  Importing the package does not
load the library; the first op call does, and raises if it is missing.
"""
