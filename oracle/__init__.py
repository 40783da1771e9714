"""fp64 CPU oracle for decode attention over a 2-/4-bit affine-quantized KV cache.

TEST INFRASTRUCTURE, NOT PRODUCT CODE. Only ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py`` may import this package. The CUDA
library never calls it and shares no code with it.

The arithmetic lives in ``oracle.c`` (plain C, compiled with gcc, built without
FMA contraction so that the single-precision quantizer rounds each operation on
its own). This module only compiles it and marshals numpy arrays through
ctypes.

Sources: "FOSCAR: Accelerating Decode Attention over 2- and 4-Bit KV Caches
through Affine Folding" (arXiv:2611.09722), abstract; and the explainer
"FOSCAR speeds up 2-bit KV decode -- Affine folding of KV dequantization"
(learnaivisually.com): receipt paragraph, quantization-format paragraph,
fold-rule paragraph, fold table, instruction-budget paragraph.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_HDR = os.path.join(_HERE, "oracle.h")
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "liboracle.so")

TOKENWISE = 0
CHANNELWISE = 1
ACC_FOLD = 0
OPERAND_FOLD = 1

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into a shared object (gcc, -O2, no FMA contraction)."""
    stale = (not os.path.exists(_SO)) or any(
        os.path.getmtime(p) > os.path.getmtime(_SO) for p in (_SRC, _HDR)
    )
    if force or stale:
        os.makedirs(_BUILD, exist_ok=True)
        tmp = _SO + f".tmp{os.getpid()}"
        cmd = [
            "gcc", "-O2", "-std=c11", "-D_GNU_SOURCE", "-ffp-contract=off", "-fno-fast-math",
            "-fPIC", "-shared", "-pthread", _SRC, "-o", tmp, "-lm",
        ]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _SO)
    return _SO


class _Args(ctypes.Structure):
    _fields_ = [
        ("B", ctypes.c_int), ("Hq", ctypes.c_int), ("Hkv", ctypes.c_int), ("D", ctypes.c_int),
        ("T_cap", ctypes.c_int), ("bits", ctypes.c_int), ("k_layout", ctypes.c_int),
        ("v_layout", ctypes.c_int), ("group", ctypes.c_int), ("sm_scale", ctypes.c_double),
        ("q", ctypes.c_void_p), ("k_codes", ctypes.c_void_p), ("k_scale", ctypes.c_void_p),
        ("k_off", ctypes.c_void_p), ("v_codes", ctypes.c_void_p), ("v_scale", ctypes.c_void_p),
        ("v_off", ctypes.c_void_p), ("seq_lens", ctypes.c_void_p), ("k_win", ctypes.c_void_p),
        ("v_win", ctypes.c_void_p), ("win_lens", ctypes.c_void_p), ("win_cap", ctypes.c_int),
        ("rotation", ctypes.c_int),
    ]


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = ctypes.CDLL(build())
            L.oracle_bf16_to_f64.restype = ctypes.c_double
            L.oracle_bf16_to_f64.argtypes = [ctypes.c_uint16]
            L.oracle_fp16_to_f64.restype = ctypes.c_double
            L.oracle_fp16_to_f64.argtypes = [ctypes.c_uint16]
            L.oracle_f64_to_fp16.restype = ctypes.c_uint16
            L.oracle_f64_to_fp16.argtypes = [ctypes.c_double]
            L.oracle_unpack_code.restype = ctypes.c_int
            L.oracle_unpack_code.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int]
            L.oracle_decode_ref.restype = ctypes.c_int
            L.oracle_decode_ref.argtypes = [ctypes.POINTER(_Args), ctypes.c_void_p, ctypes.c_int,
                                            ctypes.c_int, ctypes.c_void_p]
            L.oracle_decode_folded.restype = ctypes.c_int
            L.oracle_decode_folded.argtypes = [ctypes.POINTER(_Args), ctypes.c_int, ctypes.c_int,
                                               ctypes.c_void_p, ctypes.c_void_p]
            for name in ("oracle_weighted_dequant_sum",):
                f = getattr(L, name)
                f.restype = ctypes.c_double
                f.argtypes = [ctypes.c_void_p] * 4 + [ctypes.c_int]
            L.oracle_acc_fold.restype = ctypes.c_double
            L.oracle_acc_fold.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
                                          ctypes.c_double, ctypes.c_double]
            L.oracle_operand_fold.restype = ctypes.c_double
            L.oracle_operand_fold.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
                                              ctypes.c_void_p, ctypes.c_void_p]
            L.oracle_fold_kind.restype = ctypes.c_int
            L.oracle_fold_kind.argtypes = [ctypes.c_int, ctypes.c_int]
            L.oracle_hadamard.restype = ctypes.c_int
            L.oracle_hadamard.argtypes = [ctypes.c_int, ctypes.c_void_p]
            L.oracle_rotate_rows.restype = ctypes.c_int
            L.oracle_rotate_rows.argtypes = [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_void_p,
                                             ctypes.c_void_p]
            L.oracle_pack.restype = ctypes.c_int
            L.oracle_pack.argtypes = [ctypes.c_int] * 7 + [ctypes.c_void_p] * 5
            _lib = L
    return _lib


# ---------------------------------------------------------------- helpers

def _c(a, dtype):
    a = np.ascontiguousarray(a, dtype=dtype)
    return a, a.ctypes.data


def bf16_to_f64(h: int) -> float:
    return lib().oracle_bf16_to_f64(int(h))


def fp16_to_f64(h: int) -> float:
    return lib().oracle_fp16_to_f64(int(h))


def f64_to_fp16(x: float) -> int:
    return int(lib().oracle_f64_to_fp16(float(x)))


def unpack_code(row: np.ndarray, bits: int, d: int) -> int:
    row, p = _c(row, np.uint8)
    return int(lib().oracle_unpack_code(p, bits, d))


def weighted_dequant_sum(w, q, s, z) -> float:
    w, pw = _c(w, np.float64)
    q, pq = _c(q, np.int32)
    s, ps = _c(s, np.float64)
    z, pz = _c(z, np.float64)
    return lib().oracle_weighted_dequant_sum(pw, pq, ps, pz, len(w))


def acc_fold(w, q, s: float, z: float) -> float:
    w, pw = _c(w, np.float64)
    q, pq = _c(q, np.int32)
    return lib().oracle_acc_fold(pw, pq, len(w), float(s), float(z))


def operand_fold(w, q, s, z) -> float:
    w, pw = _c(w, np.float64)
    q, pq = _c(q, np.int32)
    s, ps = _c(s, np.float64)
    z, pz = _c(z, np.float64)
    return lib().oracle_operand_fold(pw, pq, len(w), ps, pz)


def fold_kind(side: int, layout: int) -> int:
    return int(lib().oracle_fold_kind(side, layout))


class DecodeInputs:
    """Host arrays of one decode problem in the documented layout.

    Array fields hold raw bit patterns: q, k_win, v_win as uint16 bf16 bits;
    scales and offsets as uint16 fp16 bits; codes as uint8.
    """

    def __init__(self, *, q, k_codes, k_scale, k_off, v_codes, v_scale, v_off, seq_lens,
                 bits, k_layout, v_layout, group, Hkv, T_cap, sm_scale=0.0,
                 k_win=None, v_win=None, win_lens=None, win_cap=0, rotation=0):
        self.q = np.ascontiguousarray(q, dtype=np.uint16)
        self.B, self.Hq, self.D = self.q.shape
        self.Hkv, self.T_cap = int(Hkv), int(T_cap)
        self.k_codes = np.ascontiguousarray(k_codes, dtype=np.uint8)
        self.v_codes = np.ascontiguousarray(v_codes, dtype=np.uint8)
        self.k_scale = np.ascontiguousarray(k_scale, dtype=np.uint16)
        self.k_off = np.ascontiguousarray(k_off, dtype=np.uint16)
        self.v_scale = np.ascontiguousarray(v_scale, dtype=np.uint16)
        self.v_off = np.ascontiguousarray(v_off, dtype=np.uint16)
        self.seq_lens = np.ascontiguousarray(seq_lens, dtype=np.int32)
        self.bits, self.k_layout, self.v_layout, self.group = int(bits), int(k_layout), int(v_layout), int(group)
        self.sm_scale = float(sm_scale)
        self.k_win = None if k_win is None else np.ascontiguousarray(k_win, dtype=np.uint16)
        self.v_win = None if v_win is None else np.ascontiguousarray(v_win, dtype=np.uint16)
        self.win_lens = None if win_lens is None else np.ascontiguousarray(win_lens, dtype=np.int32)
        self.win_cap = int(win_cap)
        self.rotation = int(rotation)

    def _struct(self) -> _Args:
        p = lambda a: None if a is None else a.ctypes.data  # noqa: E731
        return _Args(self.B, self.Hq, self.Hkv, self.D, self.T_cap, self.bits, self.k_layout,
                     self.v_layout, self.group, self.sm_scale, p(self.q), p(self.k_codes),
                     p(self.k_scale), p(self.k_off), p(self.v_codes), p(self.v_scale), p(self.v_off),
                     p(self.seq_lens), p(self.k_win), p(self.v_win), p(self.win_lens), self.win_cap,
                     self.rotation)


def _bits16(t) -> np.ndarray:
    import torch

    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def inputs_from_tensors(t: dict, *, bits, k_layout, v_layout, group, Hkv, T_cap, sm_scale=0.0,
                        rotation=0) -> DecodeInputs:
    """Host copies of torch tensors (q, codes, fp16 scales/offsets, seq_lens, optional window)
    as oracle inputs. Only marshalling: raw bit patterns are passed through unchanged."""
    kw = {}
    if "k_win" in t:
        kw = dict(k_win=_bits16(t["k_win"]), v_win=_bits16(t["v_win"]), win_lens=t["win_lens"].cpu().numpy(),
                  win_cap=t["k_win"].shape[2])
    return DecodeInputs(
        q=_bits16(t["q"]), k_codes=t["k_codes"].cpu().numpy(), k_scale=_bits16(t["k_scale"]),
        k_off=_bits16(t["k_off"]), v_codes=t["v_codes"].cpu().numpy(), v_scale=_bits16(t["v_scale"]),
        v_off=_bits16(t["v_off"]), seq_lens=t["seq_lens"].cpu().numpy(), bits=bits, k_layout=k_layout,
        v_layout=v_layout, group=group, Hkv=Hkv, T_cap=T_cap, sm_scale=sm_scale, rotation=rotation, **kw)


def decode_ref(x: DecodeInputs, rows=None, n_threads: int = 0) -> np.ndarray:
    """Plain definition: dequantize, textbook softmax attention. Returns fp64.

    rows: optional sequence of (b, h) pairs; the result is then [len(rows)][D],
    otherwise [B][Hq][D].
    """
    args = x._struct()
    if rows is None:
        out = np.zeros((x.B, x.Hq, x.D), dtype=np.float64)
        st = lib().oracle_decode_ref(ctypes.byref(args), None, 0, n_threads, out.ctypes.data)
    else:
        r = np.ascontiguousarray(np.asarray(rows, dtype=np.int32).reshape(-1, 2))
        out = np.zeros((r.shape[0], x.D), dtype=np.float64)
        st = lib().oracle_decode_ref(ctypes.byref(args), r.ctypes.data, r.shape[0], n_threads, out.ctypes.data)
    if st != 0:
        raise ValueError(f"oracle_decode_ref rejected the arguments (status {st})")
    return out


def attention_bf16(q_bits: np.ndarray, k_bits: np.ndarray, v_bits: np.ndarray, seq_lens, sm_scale: float = 0.0,
                   n_threads: int = 0) -> np.ndarray:
    """Plain softmax attention over a bf16 cache (the BF16 comparator's definition), fp64.

    q [B][Hq][D], k/v [B][Hkv][T][D] as uint16 bf16 bits, seq_lens [B]. It is decode_ref with
    no quantized tokens and the whole cache as the bf16 window, whose step the decode
    definition already holds (the window's tokens are attended in full precision)."""
    q = np.ascontiguousarray(q_bits, dtype=np.uint16)
    k = np.ascontiguousarray(k_bits, dtype=np.uint16)
    v = np.ascontiguousarray(v_bits, dtype=np.uint16)
    B, Hkv, T, D = k.shape
    tc = 128
    zc = np.zeros((B, Hkv, tc, D // 4), np.uint8)
    zs = np.zeros((B, Hkv, tc, D // 128), np.uint16)
    x = DecodeInputs(q=q, k_codes=zc, k_scale=zs, k_off=zs, v_codes=zc, v_scale=zs, v_off=zs,
                     seq_lens=np.zeros(B, np.int32), bits=2, k_layout=TOKENWISE, v_layout=TOKENWISE, group=128,
                     Hkv=Hkv, T_cap=tc, sm_scale=sm_scale, k_win=k, v_win=v,
                     win_lens=np.ascontiguousarray(seq_lens, dtype=np.int32), win_cap=T)
    return decode_ref(x, n_threads=n_threads)


def decode_folded(x: DecodeInputs, block: int = 64, misorder: int = 0):
    """Folded path with op counting. Returns (out [B][Hq][D] fp64, ops, values)."""
    args = x._struct()
    out = np.zeros((x.B, x.Hq, x.D), dtype=np.float64)
    ops = np.zeros(2, dtype=np.float64)
    st = lib().oracle_decode_folded(ctypes.byref(args), int(block), int(misorder), out.ctypes.data, ops.ctypes.data)
    if st != 0:
        raise ValueError(f"oracle_decode_folded rejected the arguments (status {st})")
    return out, float(ops[0]), float(ops[1])


def hadamard(n: int) -> np.ndarray:
    """Normalized Hadamard matrix of order n (fp64), from its closed form."""
    out = np.zeros((n, n), dtype=np.float64)
    if lib().oracle_hadamard(int(n), out.ctypes.data) != 0:
        raise ValueError("n must be a power of two")
    return out


def rotate_rows(x_bf16_bits: np.ndarray):
    """Rotate bf16 rows [..., n] (uint16 bits) as stored. Returns (fp32 values, bf16 bits)."""
    x, px = _c(x_bf16_bits, np.uint16)
    n = x.shape[-1]
    rows = x.size // n if n else 0
    y32 = np.zeros(x.shape, dtype=np.float32)
    y16 = np.zeros(x.shape, dtype=np.uint16)
    if lib().oracle_rotate_rows(px, rows, n, y32.ctypes.data, y16.ctypes.data) != 0:
        raise ValueError("the row length must be a power of two")
    return y32, y16


def pack(x_bf16_bits: np.ndarray, seq_lens, bits: int, layout: int, group: int,
         scale_init=None, off_init=None):
    """Quantize bf16 [B][Hkv][T_cap][D] (uint16 bits). Returns (codes, scale, off).

    scale/off start from scale_init/off_init (default zeros) so that callers can
    check that padding entries stay untouched.
    """
    x, px = _c(x_bf16_bits, np.uint16)
    B, Hkv, T_cap, D = x.shape
    sl, psl = _c(seq_lens, np.int32)
    codes = np.zeros((B, Hkv, T_cap, D * bits // 8), dtype=np.uint8)
    if layout == TOKENWISE:
        sshape = (B, Hkv, T_cap, D // group)
    else:
        sshape = (B, Hkv, T_cap // group, D)
    scale = np.zeros(sshape, np.uint16) if scale_init is None else np.array(scale_init, np.uint16).reshape(sshape)
    off = np.zeros(sshape, np.uint16) if off_init is None else np.array(off_init, np.uint16).reshape(sshape)
    st = lib().oracle_pack(B, Hkv, D, T_cap, bits, layout, group, px, psl,
                           codes.ctypes.data, scale.ctypes.data, off.ctypes.data)
    if st != 0:
        raise ValueError(f"oracle_pack rejected the arguments (status {st})")
    return codes, scale, off
