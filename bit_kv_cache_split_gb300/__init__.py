"""GB300-native decode attention over 2-/4-bit affine-quantized KV caches.

The computation lives in a CUDA library with a C ABI (include/lbkv.h); this
package builds it (``build``), binds it (``decode_attn``, ``pack``, ``append``, ``rotate``, ``decode_bf16``,
``workspace_bytes``, ``decode_launch_info``, ``alloc_workspace``, ``device_status``) and draws seeded synthetic inputs
(``inputs``).
"""

from ._binding import (CHANNELWISE, ROTATE_K, ROTATE_V, TOKENWISE, LbkvError, alloc_workspace,  # noqa: F401
                       append, decode_attn, decode_bf16, decode_launch_info, device_status, load, pack, rotate,
                       workspace_bytes)
from . import build, inputs  # noqa: F401
