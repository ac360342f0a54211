"""GB300-native (sm_103a) Engram conditional-memory forward path.

The layer (hash -> gather/dequant -> tcgen05 K/V projection -> gate -> dilated
causal conv -> residual) runs in hand-written CUDA kernels behind the C ABI of
include/engram.h; this package only marshals torch tensors into that ABI.
"""
from ._lib import EngramError, LIB_PATH  # noqa: F401
from .engram import EngramCache, EngramLayer, EngramPlan, EngramState, EngramWeights, SmSplit, stage_a_layers, stage_a_layers_e4m3  # noqa: F401
