"""ReplaySSM ring spec-verify for a Gated DeltaNet layer on GB300 (sm_103a).

The compute path is the C-ABI library libgdnspec.so (hand-written CUDA); the
Python names here only marshal arguments to it.  Importing this package does
not load the library; the first call into ``binding`` does, and fails loudly if
it is missing.
"""
