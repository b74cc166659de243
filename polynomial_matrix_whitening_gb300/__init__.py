"""ANVIL bank step on GB300 (sm_103a): twin-rail momentum, bf16 cast, Frobenius
normalisation and six quintic spectral maps on banks of projection matrices.

The compute lives in libanvil (C ABI, include/anvil.h); ``anvil`` is its thin
ctypes binding.  Import it explicitly (``from polynomial_matrix_whitening_gb300
import anvil``): it raises if the CUDA library has not been built.
"""
