"""GB300-native Megatron tensor-parallel FFN sublayer.

The computation lives in ``libtpffn.so`` (C ABI: ``include/tpffn.h``), built
from ``csrc/`` for sm_103a by ``build.build()``.  ``tpffn`` is the ctypes
binding with the ABI's names; ``ffn.TensorParallelFFN`` allocates PyTorch
buffers around it.  Import ``tpffn`` or ``ffn`` explicitly: importing them
fails loudly when the library is not built.
"""
__all__ = ["build", "tpffn", "ffn"]
