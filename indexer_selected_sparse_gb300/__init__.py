"""GB300-native indexer-selected sparse attention (QSA-style).

The compute path is the C-ABI library libqsa (hand-written sm_103a CUDA
kernels); `indexer_selected_sparse_gb300.qsa` is the thin ctypes binding over
it. Importing the package does not load the library; importing `.qsa` does,
and fails loudly if the library has not been built.
"""
