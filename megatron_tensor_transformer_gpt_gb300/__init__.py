"""GB300-native forward pass of one GPT/Llama Transformer layer as one tensor-parallel rank computes it.

The compute path is libmt_layer.so (hand-written sm_103a kernels behind a C ABI, see
include/mt_layer.h); ``mt_layer`` is its Python binding.
"""
from . import mt_layer  # noqa: F401
from .mt_layer import Layer, MtError, MtFp8Weights, MtGrads, MtWeights  # noqa: F401
