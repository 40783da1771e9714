"""The no-allocation decode entry point (lbkv_decode_attn_noalloc), called through
the C ABI, gives the same output as the regular entry point that takes a
caller-allocated workspace, on two calls in a row, and matches the fp64 oracle.

It serves callers that cannot allocate device memory at decode time (an engine
whose allocator owns all device memory, a plugin that only receives its input
and output buffers); its scratch is a fixed array inside the library, shared
by every call, so the cases below also run shapes one after another: a call
whose split counters lie where an earlier call of another shape left partials
must still start from cleared counters. This file is collected last so that a
run stopping at the first failure has already run every other test.
"""

import ctypes

import numpy as np
import pytest
import torch

import oracle
from bit_kv_cache_split_gb300 import inputs
from tests.helpers import to_oracle

pytestmark = pytest.mark.gpu

MAX_ABS = 5e-3
REL_L2 = 3e-3


def _close(got, ref):
    d = got - ref
    mx = float(np.max(np.abs(d)))
    rl2 = float(np.linalg.norm(d) / max(np.linalg.norm(ref), 1e-30))
    return mx <= MAX_ABS and rl2 <= REL_L2, mx, rl2


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import bit_kv_cache_split_gb300 as pkg
    from bit_kv_cache_split_gb300 import _binding

    pkg.build.build()
    oracle.build()
    L = _binding.load()
    assert L.lbkv_noalloc_scratch_bytes() == 16 << 20
    return L


def _noalloc(lib, wl, t):
    """One lbkv_decode_attn_noalloc call straight through ctypes; returns the fp64 output."""
    from bit_kv_cache_split_gb300 import _binding

    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    out = torch.full_like(t["q"], float("nan"))
    d = _binding.make_desc(wl.batch, wl.num_q_heads, wl.num_kv_heads, wl.t_cap)
    if wl.window:
        d.k_win, d.v_win, d.win_lens = t["k_win"].data_ptr(), t["v_win"].data_ptr(), t["win_lens"].data_ptr()
        d.win_cap = wl.window
    ptrs = [ctypes.c_void_p(t[k].data_ptr()) for k in
            ("q", "k_codes", "k_scale", "k_off", "v_codes", "v_scale", "v_off", "seq_lens")]
    st = lib.lbkv_decode_attn_noalloc(ctypes.byref(d), *ptrs, wl.bits, wl.k_layout, wl.v_layout, wl.group,
                                      ctypes.c_void_p(out.data_ptr()), stream)
    assert st == 0, _binding.strerror(st)
    torch.cuda.synchronize()
    return out.float().cpu().numpy().astype(np.float64)


def _workspace_path(t, wl):
    import bit_kv_cache_split_gb300 as pkg

    win = {}
    if wl.window:
        win = dict(k_win=t["k_win"], v_win=t["v_win"], win_lens=t["win_lens"])
    out = pkg.decode_attn(t["q"], t["k_codes"], t["k_scale"], t["k_off"], t["v_codes"], t["v_scale"], t["v_off"],
                          t["seq_lens"], bits=wl.bits, k_layout=wl.k_layout, v_layout=wl.v_layout, group=wl.group,
                          **win)
    torch.cuda.synchronize()
    return out.float().cpu().numpy().astype(np.float64)


CASES = {
    # GQA 4, group 128, token-wise K/V
    "g128-gqa4": lambda: inputs.Workload("noalloc-g128", 3, 16, 4, [700, 129, 2000], bits=2, group=128, seed=41),
    # a single long sequence first: its CTAs' partials land right after the counter region
    "b1-long": lambda: inputs.Workload("noalloc-b1", 1, 8, 2, [9000], bits=2, group=128, seed=43),
    # GQA 8, token-wise V with group 32: 32 (query, V group) columns per KV head, so the
    # plan splits each KV head into two pairs and doubles the split counters
    "g32-gqa8": lambda: inputs.Workload("noalloc-g32-gqa8", 16, 32, 4, inputs.ragged_lens(16, 300, 5000, seed=9),
                                        bits=2, group=32, seed=42),
    # a bf16 window after the cached tokens (its partials sit at the end of the scratch)
    "window": lambda: inputs.Workload("noalloc-window", 4, 16, 4, [500, 0, 1300, 77], bits=4, group=64,
                                      s_range=(0.002, 0.02), window=128, seed=44),
}


@pytest.mark.parametrize("order", [("g128-gqa4",), ("b1-long", "g32-gqa8"), ("g32-gqa8", "window", "g128-gqa4")])
def test_noalloc_entry_point_matches_workspace_entry_point_and_oracle(lib, order):
    """Shapes run back to back through the shared scratch; each one twice in a row."""
    for name in order:
        wl = CASES[name]()
        host = inputs.generate(wl, "cpu")
        t = {k: v.cuda() for k, v in host.items()}
        ref_ws = _workspace_path(t, wl)
        ref = oracle.decode_ref(to_oracle(host, wl))
        outs = []
        for call in range(2):
            got = _noalloc(lib, wl, t)
            assert np.all(np.isfinite(got)), f"{name} call {call}: non-finite output"
            ok, mx, rl2 = _close(got, ref)
            assert ok, f"{name} call {call} against the oracle: max-abs {mx:.3e}, rel-L2 {rl2:.3e}"
            ok, mx, rl2 = _close(got, ref_ws)
            assert ok, f"{name} call {call} against the workspace entry point: max-abs {mx:.3e}, rel-L2 {rl2:.3e}"
            outs.append(got)
        ok, mx, rl2 = _close(outs[1], outs[0])
        assert ok, f"{name} second call: max-abs {mx:.3e}, rel-L2 {rl2:.3e}"


def test_noalloc_rejects_scratch_beyond_the_array(lib):
    from bit_kv_cache_split_gb300 import _binding

    # With a bf16 window, 4096 sequences x 64 query heads need one window partial per
    # (sequence, KV head): far more than 16 MiB. The call is rejected before any pointer
    # is touched (the window pointers below are never dereferenced) or anything launched.
    d = _binding.make_desc(4096, 64, 8, 1 << 20)
    d.k_win = d.v_win = d.win_lens = 4096
    d.win_cap = 128
    null = ctypes.c_void_p(0)
    st = lib.lbkv_decode_attn_noalloc(ctypes.byref(d), *([null] * 8), 2, 0, 0, 128, null, null)
    assert st == -7
    assert b"scratch" in lib.lbkv_strerror(st)
