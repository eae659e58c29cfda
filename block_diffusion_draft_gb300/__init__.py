"""GB300-native DFlash draft attention: a C-ABI CUDA library for sm_103a
(include/dflash_attn.h) and its thin Python binding."""
from .dflash_attn import (DFlashAttention, DFlashError, DraftCache,  # noqa: F401
                          DecoderMLP, KVGroup, PagedCache, declared_functions, lib)
