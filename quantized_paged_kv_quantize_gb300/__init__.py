"""GB300-native quantized paged KV cache: quantize-on-write and fused-dequant
paged decode attention (libkvq, sm_103a).  ``kvq`` is the binding of the C ABI
declared in include/kvq.h."""
from . import kvq  # noqa: F401  (raises ImportError if libkvq.so is missing)

__all__ = ["kvq"]
