"""Block-quantized wire codec for GB300 (sm_103a).

Importing the package loads nothing; the CUDA library ``libbq.so`` is loaded the
first time a codec call is made, and a missing or unbuildable library raises
instead of falling back to any other implementation.
"""
