"""Thin ctypes binding of the C ABI in include/lbkv.h.

Argument marshalling only: tensors are checked for device, dtype, shape and
contiguity and passed as raw pointers with the current CUDA stream. Every step
of the computation runs in the CUDA library; if the library is missing this
module raises instead of falling back to anything else.
"""

from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

import torch

from . import build as _build

TOKENWISE = 0
CHANNELWISE = 1
ROTATE_K = 1  # keys stored rotated by the normalized Hadamard matrix (lbkv_rotation)
ROTATE_V = 2  # values stored rotated

STATUS = {0: "LBKV_OK", -1: "LBKV_EINVAL", -2: "LBKV_EALIGN", -3: "LBKV_EUNSUPPORTED",
          -4: "LBKV_EWORKSPACE", -5: "LBKV_ECUDA", -6: "LBKV_EDEVICE", -7: "LBKV_ESCRATCH"}

EXPORTS = ("lbkv_workspace_bytes", "lbkv_decode_attn", "lbkv_pack", "lbkv_append", "lbkv_decode_bf16",
           "lbkv_bf16_workspace_bytes", "lbkv_rotate", "lbkv_device_status",
           "lbkv_strerror", "lbkv_decode_attn_noalloc", "lbkv_noalloc_scratch_bytes", "lbkv_selftest_wait_timeout")


class LbkvError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS.get(status, status)} ({strerror(status)})")


class Desc(ctypes.Structure):
    """Mirror of lbkv_desc."""

    _fields_ = [
        ("batch", ctypes.c_int32), ("num_q_heads", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32), ("max_seq_len", ctypes.c_int32), ("sm_scale", ctypes.c_float),
        ("k_win", ctypes.c_void_p), ("v_win", ctypes.c_void_p), ("win_lens", ctypes.c_void_p),
        ("win_cap", ctypes.c_int32), ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t),
        ("page_table", ctypes.c_void_p), ("page_tokens", ctypes.c_int32), ("max_pages", ctypes.c_int32),
        ("num_pages", ctypes.c_int32), ("rotation", ctypes.c_int32),
    ]


_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return _build.LIB


def load(path: Optional[str] = None):
    """Load liblbkv.so (built by bit_kv_cache_split_gb300.build.build()); raise if absent."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or library_path()
        if not os.path.exists(p):
            raise RuntimeError(f"CUDA library {p} is missing; run bit_kv_cache_split_gb300.build.build() first")
        L = ctypes.CDLL(p)
        vp, i32 = ctypes.c_void_p, ctypes.c_int
        L.lbkv_workspace_bytes.restype = ctypes.c_size_t
        L.lbkv_workspace_bytes.argtypes = [ctypes.POINTER(Desc), i32, i32, i32, i32]
        L.lbkv_decode_attn.restype = i32
        L.lbkv_decode_attn.argtypes = [ctypes.POINTER(Desc)] + [vp] * 8 + [i32] * 4 + [vp, vp]
        L.lbkv_pack.restype = i32
        L.lbkv_pack.argtypes = [ctypes.POINTER(Desc), vp, vp, i32, i32, i32, vp, vp, vp, vp]
        L.lbkv_decode_bf16.restype = i32
        L.lbkv_decode_bf16.argtypes = [ctypes.POINTER(Desc)] + [vp] * 6
        L.lbkv_bf16_workspace_bytes.restype = ctypes.c_size_t
        L.lbkv_bf16_workspace_bytes.argtypes = [ctypes.POINTER(Desc)]
        L.lbkv_append.restype = i32
        L.lbkv_append.argtypes = [ctypes.POINTER(Desc), vp, vp, vp] + [i32] * 4 + [vp] * 7
        L.lbkv_rotate.restype = i32
        L.lbkv_rotate.argtypes = [vp, vp, ctypes.c_int64, i32, vp]
        L.lbkv_selftest_wait_timeout.restype = i32
        L.lbkv_selftest_wait_timeout.argtypes = [vp, ctypes.c_uint64, vp]
        L.lbkv_device_status.restype = i32
        L.lbkv_device_status.argtypes = [ctypes.POINTER(Desc), vp, ctypes.POINTER(ctypes.c_int32)]
        L.lbkv_decode_attn_noalloc.restype = i32
        L.lbkv_decode_attn_noalloc.argtypes = [ctypes.POINTER(Desc)] + [vp] * 8 + [i32] * 4 + [vp, vp]
        L.lbkv_noalloc_scratch_bytes.restype = ctypes.c_size_t
        L.lbkv_noalloc_scratch_bytes.argtypes = []
        L.lbkv_decode_launch_info.restype = i32
        L.lbkv_decode_launch_info.argtypes = [ctypes.POINTER(Desc)] + [i32] * 4 + [ctypes.POINTER(ctypes.c_int)] * 3
        L.lbkv_strerror.restype = ctypes.c_char_p
        L.lbkv_strerror.argtypes = [i32]
        if path is None:
            _lib = L
        return L


def strerror(status: int) -> str:
    try:
        return load().lbkv_strerror(int(status)).decode()
    except RuntimeError:
        return STATUS.get(status, "unknown")


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_ptr(stream) -> ctypes.c_void_p:
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _check(t: torch.Tensor, name: str, dtype, shape=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device.type != "cuda":
        raise ValueError(f"{name} must be on a CUDA device")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


def make_desc(batch, num_q_heads, num_kv_heads, max_seq_len, head_dim=128, sm_scale=0.0, k_win=None,
              v_win=None, win_lens=None, workspace=None) -> Desc:
    d = Desc()
    d.batch, d.num_q_heads, d.num_kv_heads = int(batch), int(num_q_heads), int(num_kv_heads)
    d.head_dim, d.max_seq_len, d.sm_scale = int(head_dim), int(max_seq_len), float(sm_scale)
    d.k_win = None if k_win is None else k_win.data_ptr()
    d.v_win = None if v_win is None else v_win.data_ptr()
    d.win_lens = None if win_lens is None else win_lens.data_ptr()
    d.win_cap = 0 if k_win is None else int(k_win.shape[2])
    d.workspace = None if workspace is None else workspace.data_ptr()
    d.workspace_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    return d


def _set_paged(d: Desc, page_table, page_tokens: int, num_pages: int):
    """Paged-cache fields of d: page_table int32 [B][max_pages] on the device."""
    _check(page_table, "page_table", torch.int32)
    if page_table.dim() != 2 or page_table.shape[0] != d.batch:
        raise ValueError(f"page_table must have shape ({d.batch}, max_pages), got {tuple(page_table.shape)}")
    d.page_table = page_table.data_ptr()
    d.page_tokens, d.max_pages, d.num_pages = int(page_tokens), int(page_table.shape[1]), int(num_pages)


def _cache_shape(B, Hkv, T, page_table, page_tokens, num_pages):
    """Leading dims of the cache tensors: [B][Hkv][T] contiguous, [num_pages][Hkv][page_tokens] paged."""
    return (B, Hkv, T) if page_table is None else (num_pages, Hkv, page_tokens)


def _paged_dims(k_codes, page_table, max_seq_len):
    """(num_pages, page_tokens, max_seq_len) of a paged cache, read from the code pool and the table."""
    NP, P = k_codes.shape[0], k_codes.shape[2]
    T = int(max_seq_len) if max_seq_len else int(page_table.shape[1]) * P
    return NP, P, T


def workspace_bytes(batch, num_q_heads, num_kv_heads, max_seq_len, bits, k_layout, v_layout, group,
                    window: bool = False, head_dim=128) -> int:
    """Workspace size for a call with these shapes (0 when the arguments are invalid)."""
    d = make_desc(batch, num_q_heads, num_kv_heads, max_seq_len, head_dim)
    if window:
        d.k_win = d.v_win = d.win_lens = 16  # any non-null value: only presence matters here
        d.win_cap = 1
    return int(load().lbkv_workspace_bytes(ctypes.byref(d), bits, k_layout, v_layout, group))


def decode_launch_info(batch, num_q_heads, num_kv_heads, max_seq_len, bits, k_layout=TOKENWISE, v_layout=TOKENWISE,
                       group=128, window: bool = False, paged_tokens: int = 0, head_dim=128) -> dict:
    """The launch lbkv_decode_launch_info reports for a call with these shapes on the current
    device: {"grid": CTAs, "cluster": CTAs per cluster (0: the split-decode grid), "split":
    clusters per (sequence, KV head) pair}. Raises LbkvError for invalid arguments."""
    d = make_desc(batch, num_q_heads, num_kv_heads, max_seq_len, head_dim)
    if window:
        d.k_win = d.v_win = d.win_lens = 16  # any non-null value: only presence matters here
        d.win_cap = 1
    if paged_tokens:
        d.page_table = 16
        d.page_tokens = paged_tokens
        d.max_pages = max(1, max_seq_len // paged_tokens)
        d.num_pages = d.max_pages * max(1, batch)
    g, c, s = ctypes.c_int(0), ctypes.c_int(0), ctypes.c_int(0)
    st = load().lbkv_decode_launch_info(ctypes.byref(d), bits, k_layout, v_layout, group, ctypes.byref(g),
                                        ctypes.byref(c), ctypes.byref(s))
    if st != 0:
        raise LbkvError(st, "lbkv_decode_launch_info")
    return {"grid": g.value, "cluster": c.value, "split": s.value}


def alloc_workspace(nbytes: int, device) -> torch.Tensor:
    """Zero-filled byte tensor, 256-byte aligned (torch's allocator aligns to 512)."""
    ws = torch.zeros(max(nbytes, 256), dtype=torch.uint8, device=device)
    assert ws.data_ptr() % 256 == 0
    return ws


def decode_attn(q, k_codes, k_scale, k_off, v_codes, v_scale, v_off, seq_lens, *, bits, k_layout=TOKENWISE,
                v_layout=TOKENWISE, group=128, sm_scale=0.0, k_win=None, v_win=None, win_lens=None,
                page_table=None, max_seq_len=None, rotation=0, out=None, workspace=None,
                stream=None) -> torch.Tensor:
    """Decode attention through lbkv_decode_attn. Shapes as in include/lbkv.h.

    q bf16 [B][Hq][D]; k_codes/v_codes uint8 [B][Hkv][T_cap][D*bits/8]; scales/offsets fp16;
    seq_lens int32 [B] on the device. Returns out bf16 [B][Hq][D] (allocated when not given).
    Paged cache: page_table int32 [B][max_pages]; the cache tensors are page pools
    ([num_pages][Hkv][page_tokens]...) and max_seq_len defaults to max_pages * page_tokens.
    rotation: ROTATE_K | ROTATE_V bits of a cache (and window) stored rotated (see rotate).
    """
    B, Hq, D = q.shape
    Hkv, T = k_codes.shape[1], k_codes.shape[2]
    NP = P = 0
    if page_table is not None:
        NP, P, T = _paged_dims(k_codes, page_table, max_seq_len)
    _check(q, "q", torch.bfloat16)
    for name, t in (("k_codes", k_codes), ("v_codes", v_codes)):
        _check(t, name, torch.uint8, _cache_shape(B, Hkv, T, page_table, P, NP) + (D * bits // 8,))
    for name, t in (("k_scale", k_scale), ("k_off", k_off), ("v_scale", v_scale), ("v_off", v_off)):
        _check(t, name, torch.float16)
    _check(seq_lens, "seq_lens", torch.int32, (B,))
    if k_win is not None:
        _check(k_win, "k_win", torch.bfloat16)
        _check(v_win, "v_win", torch.bfloat16, tuple(k_win.shape))
        _check(win_lens, "win_lens", torch.int32, (B,))
    if out is None:
        out = torch.empty((B, Hq, D), dtype=torch.bfloat16, device=q.device)
    _check(out, "out", torch.bfloat16, (B, Hq, D))
    L = load()
    if workspace is None:
        n = workspace_bytes(B, Hq, Hkv, T, bits, k_layout, v_layout, group, window=k_win is not None)
        if n == 0:
            raise LbkvError(-3 if bits in (2, 4) else -1, "lbkv_workspace_bytes")
        workspace = alloc_workspace(n, q.device)
    d = make_desc(B, Hq, Hkv, T, D, sm_scale, k_win, v_win, win_lens, workspace)
    d.rotation = int(rotation)
    if page_table is not None:
        _set_paged(d, page_table, P, NP)
    st = L.lbkv_decode_attn(ctypes.byref(d), _ptr(q), _ptr(k_codes), _ptr(k_scale), _ptr(k_off), _ptr(v_codes),
                            _ptr(v_scale), _ptr(v_off), _ptr(seq_lens), int(bits), int(k_layout), int(v_layout),
                            int(group), _ptr(out), _stream_ptr(stream))
    if st != 0:
        raise LbkvError(st, "lbkv_decode_attn")
    return out


def pack(x, seq_lens, *, bits, layout=TOKENWISE, group=128, codes=None, scale=None, off=None, page_table=None,
         num_pages=None, page_tokens=None, workspace=None, stream=None):
    """Quantize bf16 x [B][Hkv][T_cap][D] through lbkv_pack. Returns (codes, scale, off).

    Paged cache: page_table int32 [B][max_pages]; codes, scale and off are page pools
    [num_pages][Hkv][page_tokens]... (allocated zero-filled from num_pages and page_tokens
    when not given); workspace (optional) receives the device status."""
    _check(x, "x", torch.bfloat16)
    B, Hkv, T, D = x.shape
    _check(seq_lens, "seq_lens", torch.int32, (B,))
    if page_table is not None and codes is not None:
        num_pages, page_tokens = codes.shape[0], codes.shape[2]
    lead = _cache_shape(B, Hkv, T, page_table, page_tokens, num_pages)
    R = lead[2]
    sshape = lead + (D // group,) if layout == TOKENWISE else lead[:2] + (R // group, D)
    if codes is None:
        alloc = torch.empty if page_table is None else torch.zeros
        codes = alloc(lead + (D * bits // 8,), dtype=torch.uint8, device=x.device)
    if scale is None:
        scale = torch.zeros(sshape, dtype=torch.float16, device=x.device)
    if off is None:
        off = torch.zeros(sshape, dtype=torch.float16, device=x.device)
    _check(codes, "codes", torch.uint8, lead + (D * bits // 8,))
    _check(scale, "scale", torch.float16, sshape)
    _check(off, "off", torch.float16, sshape)
    d = make_desc(B, 1, Hkv, T, D, workspace=workspace)
    d.num_q_heads = Hkv
    if page_table is not None:
        _set_paged(d, page_table, page_tokens, num_pages)
    st = load().lbkv_pack(ctypes.byref(d), _ptr(x), _ptr(seq_lens), int(bits), int(layout), int(group),
                          _ptr(codes), _ptr(scale), _ptr(off), _stream_ptr(stream))
    if st != 0:
        raise LbkvError(st, "lbkv_pack")
    return codes, scale, off


def append(k_new, v_new, seq_lens, k_codes, k_scale, k_off, v_codes, v_scale, v_off, *, bits, k_layout=TOKENWISE,
           v_layout=TOKENWISE, group=128, k_win=None, v_win=None, win_lens=None, page_table=None, max_seq_len=None,
           rotation=0, workspace=None, stream=None):
    """Append the new token k_new/v_new bf16 [B][Hkv][D] through lbkv_append (quantize-on-append).

    The cache tensors, seq_lens (and win_lens with the window) are updated in place. Paged
    cache: page_table int32 [B][max_pages] and page pools, as for decode_attn. rotation: the sides
    stored rotated (ROTATE_K | ROTATE_V), rotated on the way in."""
    _check(k_new, "k_new", torch.bfloat16)
    B, Hkv, D = k_new.shape
    _check(v_new, "v_new", torch.bfloat16, (B, Hkv, D))
    _check(seq_lens, "seq_lens", torch.int32, (B,))
    T = k_codes.shape[2]
    NP = P = 0
    if page_table is not None:
        NP, P, T = _paged_dims(k_codes, page_table, max_seq_len)
    for name, t in (("k_codes", k_codes), ("v_codes", v_codes)):
        _check(t, name, torch.uint8, _cache_shape(B, Hkv, T, page_table, P, NP) + (D * bits // 8,))
    for name, t in (("k_scale", k_scale), ("k_off", k_off), ("v_scale", v_scale), ("v_off", v_off)):
        _check(t, name, torch.float16)
    if k_win is not None:
        _check(k_win, "k_win", torch.bfloat16)
        _check(v_win, "v_win", torch.bfloat16, tuple(k_win.shape))
        _check(win_lens, "win_lens", torch.int32, (B,))
    d = make_desc(B, Hkv, Hkv, T, D, k_win=k_win, v_win=v_win, win_lens=win_lens, workspace=workspace)
    d.rotation = int(rotation)
    if page_table is not None:
        _set_paged(d, page_table, P, NP)
    st = load().lbkv_append(ctypes.byref(d), _ptr(k_new), _ptr(v_new), _ptr(seq_lens), int(bits), int(k_layout),
                            int(v_layout), int(group), _ptr(k_codes), _ptr(k_scale), _ptr(k_off), _ptr(v_codes),
                            _ptr(v_scale), _ptr(v_off), _stream_ptr(stream))
    if st != 0:
        raise LbkvError(st, "lbkv_append")


def rotate(x, out=None, stream=None):
    """Rows of bf16 x [..., 128] rotated by the normalized Hadamard matrix (lbkv_rotate):
    the step that stores a cache rotated. out may be x itself (in place)."""
    _check(x, "x", torch.bfloat16)
    if out is None:
        out = torch.empty_like(x)
    _check(out, "out", torch.bfloat16, tuple(x.shape))
    D = x.shape[-1] if x.dim() else 0
    rows = x.numel() // D if D else 0
    st = load().lbkv_rotate(_ptr(x), _ptr(out), int(rows), int(D), _stream_ptr(stream))
    if st != 0:
        raise LbkvError(st, "lbkv_rotate")
    return out


def decode_bf16(q, k, v, seq_lens, *, sm_scale=0.0, out=None, workspace=None, stream=None):
    """The BF16 comparator (lbkv_decode_bf16): decode attention over bf16 k, v [B][Hkv][T][D]."""
    _check(q, "q", torch.bfloat16)
    B, Hq, D = q.shape
    _check(k, "k", torch.bfloat16)
    Hkv, T = k.shape[1], k.shape[2]
    _check(k, "k", torch.bfloat16, (B, Hkv, T, D))
    _check(v, "v", torch.bfloat16, (B, Hkv, T, D))
    _check(seq_lens, "seq_lens", torch.int32, (B,))
    if out is None:
        out = torch.empty((B, Hq, D), dtype=torch.bfloat16, device=q.device)
    _check(out, "out", torch.bfloat16, (B, Hq, D))
    d = make_desc(B, Hq, Hkv, T, D, sm_scale=sm_scale)
    L = load()
    if workspace is None:
        n = L.lbkv_bf16_workspace_bytes(ctypes.byref(d))
        if n == 0:
            raise LbkvError(-3, "lbkv_bf16_workspace_bytes")
        workspace = torch.zeros(n, dtype=torch.uint8, device=q.device)
    d.workspace = workspace.data_ptr()
    d.workspace_bytes = workspace.numel() * workspace.element_size()
    st = L.lbkv_decode_bf16(ctypes.byref(d), _ptr(q), _ptr(k), _ptr(v), _ptr(seq_lens), _ptr(out),
                            _stream_ptr(stream))
    if st != 0:
        raise LbkvError(st, "lbkv_decode_bf16")
    return out


def selftest_wait_timeout(limit_ns: int, device="cuda") -> tuple:
    """Run the bounded-wait self-test (lbkv_selftest_wait_timeout) and return the two
    status words (the recorded code, and how many warps went on past the failed wait)."""
    s = torch.zeros(4, dtype=torch.int32, device=device)
    st = load().lbkv_selftest_wait_timeout(s.data_ptr(), int(limit_ns), _stream_ptr(None))
    if st != 0:
        raise LbkvError(st, "lbkv_selftest_wait_timeout")
    torch.cuda.synchronize()
    return int(s[0].item()), int(s[1].item())


def device_status(workspace: torch.Tensor, stream=None) -> int:
    """Read and clear the device status word (synchronizes the stream). Returns the code (0 = fine)."""
    d = Desc()
    d.workspace = workspace.data_ptr()
    d.workspace_bytes = workspace.numel() * workspace.element_size()
    code = ctypes.c_int32(0)
    st = load().lbkv_device_status(ctypes.byref(d), _stream_ptr(stream), ctypes.byref(code))
    if st not in (0, -6):
        raise LbkvError(st, "lbkv_device_status")
    return int(code.value)
