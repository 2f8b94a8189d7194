"""GB300-native 4-bit group-symmetric weight-quantized linear (q4gsw / qcs4w).

out[m,n] = bias[n] + sum_k x[m,k] * (nib(W)[n,k] - 8) * scale[k / group_size, n]

The compute path is the C-ABI library ``libq4lin.so`` (hand-written sm_103a CUDA
kernels); ``q4lin`` is its thin ctypes binding.  ``synth`` draws seeded inputs.
"""
