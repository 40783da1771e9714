"""GB300-native decode attention over 2-/4-bit affine-quantized KV caches.

The computation lives in a CUDA library with a C ABI (include/lbkv.h); this
package builds it (``build``), binds it (``decode_attn``, ``pack``, ``append``,
``workspace_bytes``, ``device_status``) and draws seeded synthetic inputs
(``inputs``).
"""

from ._binding import (CHANNELWISE, TOKENWISE, LbkvError, append, decode_attn, device_status, load, pack,  # noqa: F401
                       workspace_bytes)
from . import build, inputs  # noqa: F401
