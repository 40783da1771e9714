"""GB300-native decode attention over 2-/4-bit affine-quantized KV caches.

The computation lives in a CUDA library with a C ABI (include/lbkv.h); this
package builds it (``build``), binds it (``decode_attn``, ``pack``, ``append``, ``decode_bf16``,
``workspace_bytes``, ``device_status``) and draws seeded synthetic inputs
(``inputs``).
"""

from ._binding import (CHANNELWISE, TOKENWISE, LbkvError, append, decode_attn, decode_bf16,  # noqa: F401
                       device_status, load, pack, workspace_bytes)
from . import build, inputs  # noqa: F401
