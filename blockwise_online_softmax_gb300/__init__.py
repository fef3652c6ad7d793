"""GB300-native blockwise online-softmax (Ring Attention forward) library.

The compute path is ``libra.so``, a C-ABI library of hand-written sm_103a
CUDA kernels.  ``binding`` marshals torch tensors into it.  Importing this
package does not load the library.  The first call of a binding function
loads it, and raises if it has not been built.
"""
