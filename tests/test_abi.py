"""Host-side checks of the C ABI that need no GPU: the library builds, loads,
exports every function include/lbkv.h declares, and rejects invalid arguments
before touching the device."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from bit_kv_cache_split_gb300 import _binding, build

    build.build()
    return _binding.load()


def declared_functions():
    names = []
    inc = os.path.join(ROOT, "include")
    for f in sorted(os.listdir(inc)):
        if f.endswith(".h"):
            with open(os.path.join(inc, f)) as fh:
                text = fh.read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names += re.findall(r"^\s*LBKV_API\s+[\w\s\*]+?\b(lbkv_\w+)\s*\(", text, flags=re.M)
    return names


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("lbkv_decode_attn", "lbkv_pack", "lbkv_workspace_bytes", "lbkv_strerror", "lbkv_device_status"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert names
    for n in names:
        assert hasattr(lib, n), n


def test_strerror_texts(lib):
    from bit_kv_cache_split_gb300 import _binding

    for st in _binding.STATUS:
        assert lib.lbkv_strerror(st)
    assert lib.lbkv_strerror(0) == b"success"
    assert b"unknown" in lib.lbkv_strerror(12345)


def _desc(**kw):
    from bit_kv_cache_split_gb300 import _binding

    d = _binding.make_desc(kw.pop("B", 1), kw.pop("Hq", 32), kw.pop("Hkv", 8), kw.pop("T", 4096),
                           kw.pop("D", 128))
    for k, v in kw.items():
        setattr(d, k, v)
    return d


@pytest.mark.parametrize("kwargs,fmt,want", [
    (dict(), (3, 0, 0, 128), -1),              # bits
    (dict(), (2, 2, 0, 128), -1),              # layout
    (dict(), (2, 0, 0, 16), -3),               # group
    (dict(D=64), (2, 0, 0, 128), -3),          # head_dim
    (dict(Hq=30, Hkv=8), (2, 0, 0, 128), -1),  # Hq % Hkv
    (dict(Hq=24, Hkv=8), (2, 0, 0, 128), -3),  # Hq/Hkv = 3
    (dict(T=1000), (2, 0, 0, 128), -1),        # T_cap not a multiple of 128
    (dict(T=0), (2, 0, 0, 128), -1),
    (dict(B=-1), (2, 0, 0, 128), -1),
])
def test_invalid_decode_arguments_rejected_before_launch(lib, kwargs, fmt, want):
    d = _desc(**kwargs)
    null = ctypes.c_void_p(0)
    st = lib.lbkv_decode_attn(ctypes.byref(d), *([null] * 8), *fmt, null, null)
    assert st == want
    assert lib.lbkv_workspace_bytes(ctypes.byref(d), *fmt) == 0


@pytest.mark.parametrize("hq,fmt", [(4, (2, 0, 0, 32)), (8, (2, 0, 0, 64)), (8, (4, 1, 0, 64)), (1, (4, 0, 0, 32)),
                                    (8, (2, 0, 0, 32)), (8, (4, 1, 0, 32))])
def test_tokenwise_v_group_combinations_supported(lib, hq, fmt):
    """Up to 16 (query, value channel group) pairs per KV head are supported."""
    d = _desc(Hq=8 * hq, Hkv=8)
    null = ctypes.c_void_p(0)
    # past the format checks: a machine without a GPU stops at the device query, one with
    # a GPU at the NULL pointers; neither answers "unsupported"
    assert lib.lbkv_decode_attn(ctypes.byref(d), *([null] * 8), *fmt, null, null) not in (0, -3)


def test_window_arguments_validated(lib):
    d = _desc()
    d.k_win = 4096  # v_win and win_lens left NULL
    null = ctypes.c_void_p(0)
    assert lib.lbkv_decode_attn(ctypes.byref(d), *([null] * 8), 2, 0, 0, 128, null, null) == -1
    d.v_win = d.win_lens = 4096
    d.win_cap = 129
    assert lib.lbkv_decode_attn(ctypes.byref(d), *([null] * 8), 2, 0, 0, 128, null, null) == -1


@pytest.mark.parametrize("fmt,want", [((3, 0, 128), -1), ((2, 5, 128), -1), ((2, 0, 100), -3)])
def test_invalid_pack_arguments_rejected(lib, fmt, want):
    d = _desc()
    null = ctypes.c_void_p(0)
    assert lib.lbkv_pack(ctypes.byref(d), null, null, *fmt, null, null, null, null) == want


@pytest.mark.parametrize("kwargs,fmt,want", [
    (dict(), (3, 0, 0, 128), -1),              # bits
    (dict(), (2, 0, 0, 16), -3),               # group
    (dict(Hq=24, Hkv=8), (2, 0, 0, 128), -3),  # Hq/Hkv = 3
    (dict(T=1000), (2, 0, 0, 128), -1),        # T_cap not a multiple of 128
])
def test_launch_info_rejects_what_decode_rejects(lib, kwargs, fmt, want):
    d = _desc(**kwargs)
    g, c, s = ctypes.c_int(-7), ctypes.c_int(-7), ctypes.c_int(-7)
    assert lib.lbkv_decode_launch_info(ctypes.byref(d), *fmt, ctypes.byref(g), ctypes.byref(c), ctypes.byref(s)) == want
    null = ctypes.c_void_p(0)
    assert lib.lbkv_decode_attn(ctypes.byref(d), *([null] * 8), *fmt, null, null) == want


def test_launch_info_needs_its_outputs(lib):
    d = _desc()
    g = ctypes.c_int(0)
    assert lib.lbkv_decode_launch_info(ctypes.byref(d), 2, 0, 0, 128, ctypes.byref(g), None, None) == -1
    assert lib.lbkv_decode_launch_info(None, 2, 0, 0, 128, ctypes.byref(g), ctypes.byref(g), ctypes.byref(g)) == -1


def test_null_descriptor(lib):
    null = ctypes.c_void_p(0)
    assert lib.lbkv_decode_attn(None, *([null] * 8), 2, 0, 0, 128, null, null) == -1
    assert lib.lbkv_pack(None, null, null, 2, 0, 128, null, null, null, null) == -1
    assert lib.lbkv_workspace_bytes(None, 2, 0, 0, 128) == 0
    assert lib.lbkv_device_status(None, null, None) == -1


def test_empty_batch_is_a_no_op_without_pointers(lib):
    # B = 0 validates the shapes and returns before any launch; a GPU-less host
    # can still reject it with LBKV_ECUDA when the device cannot be queried.
    d = _desc(B=0)
    null = ctypes.c_void_p(0)
    assert lib.lbkv_decode_attn(ctypes.byref(d), *([null] * 8), 2, 0, 0, 128, null, null) in (0, -5)
    assert lib.lbkv_pack(ctypes.byref(d), null, null, 2, 0, 128, null, null, null, null) == 0


@pytest.mark.parametrize("status,limit,want", [(0, 1000, -1), (4096, 0, -1), (4096, 2_000_000_000, -1), (4100, 1000, -2)])
def test_selftest_arguments_rejected_before_launch(lib, status, limit, want):
    assert lib.lbkv_selftest_wait_timeout(ctypes.c_void_p(status), ctypes.c_uint64(limit), ctypes.c_void_p(0)) == want



def _append(lib, d, fmt, ptrs=None):
    null = ctypes.c_void_p(0)
    p = ptrs if ptrs is not None else [null] * 3
    return lib.lbkv_append(ctypes.byref(d) if d is not None else None, *p, *fmt, *([null] * 6), null)


@pytest.mark.parametrize("kwargs,fmt,want", [
    (dict(), (3, 0, 0, 128), -1),        # bits
    (dict(), (2, 0, 2, 128), -1),        # layout
    (dict(), (2, 0, 0, 16), -3),         # group
    (dict(D=64), (2, 0, 0, 128), -3),    # head_dim
    (dict(T=1000), (2, 0, 0, 128), -1),  # T_cap not a multiple of 128
    (dict(B=-1), (2, 0, 0, 128), -1),
    (dict(), (2, 1, 0, 128), -1),        # a channel-wise side needs the window
    (dict(), (2, 0, 0, 128), -1),        # null pointers
])
def test_invalid_append_arguments_rejected_before_launch(lib, kwargs, fmt, want):
    assert _append(lib, _desc(**kwargs), fmt) == want


def test_append_window_rules(lib):
    # the window must hold a whole channel-wise group, and all three window fields go together
    d = _desc()
    d.k_win = d.v_win = d.win_lens = 4096
    d.win_cap = 64
    assert _append(lib, d, (2, 1, 0, 128)) == -1
    d.win_cap = 128
    assert _append(lib, d, (2, 1, 0, 128)) == -1  # past the window rules: null cache pointers
    d.v_win = None
    assert _append(lib, d, (2, 0, 1, 64)) == -1
    assert _append(lib, None, (2, 0, 0, 128)) == -1


def test_append_misaligned_pointer(lib):
    d = _desc()
    ok, bad = ctypes.c_void_p(4096), ctypes.c_void_p(4100)
    st = lib.lbkv_append(ctypes.byref(d), ok, bad, ok, 2, 0, 0, 128, *([ok] * 6), ctypes.c_void_p(0))
    assert st == -2


def test_append_empty_batch_is_a_no_op(lib):
    assert _append(lib, _desc(B=0), (2, 0, 0, 128)) == 0


@pytest.mark.parametrize("args,want", [
    ((4096, 4096, -1, 128), -1),     # negative row count
    ((4096, 4096, 8, 64), -3),       # head_dim
    ((0, 4096, 8, 128), -1),         # null input
    ((4096, 0, 8, 128), -1),         # null output
    ((4100, 4096, 8, 128), -2),      # misaligned
    ((0, 0, 0, 128), 0),             # no rows: nothing to do
])
def test_rotate_arguments_rejected_before_launch(lib, args, want):
    x, y, rows, d = args
    assert lib.lbkv_rotate(ctypes.c_void_p(x), ctypes.c_void_p(y), ctypes.c_int64(rows), d, ctypes.c_void_p(0)) == want


def test_rotation_flags_validated(lib):
    null = ctypes.c_void_p(0)
    d = _desc()
    d.rotation = 4  # no such bit
    assert lib.lbkv_decode_attn(ctypes.byref(d), *([null] * 8), 2, 0, 0, 128, null, null) == -1
    assert lib.lbkv_workspace_bytes(ctypes.byref(d), 2, 0, 0, 128) == 0
    assert lib.lbkv_append(ctypes.byref(d), null, null, null, 2, 0, 0, 128, *([null] * 6), null) == -1
    d.rotation = 3  # the comparator reads a plain bf16 cache only
    assert lib.lbkv_bf16_workspace_bytes(ctypes.byref(d)) == 0
    assert lib.lbkv_decode_bf16(ctypes.byref(d), *([null] * 5), null) == -3
    # a valid flag passes the format checks (a GPU-less host stops at the device query)
    assert lib.lbkv_decode_attn(ctypes.byref(d), *([null] * 8), 2, 0, 0, 128, null, null) not in (0, -1, -3)
