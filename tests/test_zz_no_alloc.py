"""The no-allocation decode entry point (lbkv_decode_attn_noalloc), called through
the C ABI, gives the same output as the regular entry point that takes a
caller-allocated workspace, on two calls in a row.

It serves callers that cannot allocate device memory at decode time (an engine
whose allocator owns all device memory, a plugin that only receives its input
and output buffers); its scratch is a fixed array inside the library. This file
is collected last so that a run stopping at the first failure has already run
every other test.
"""

import ctypes

import numpy as np
import pytest
import torch

from bit_kv_cache_split_gb300 import inputs

pytestmark = pytest.mark.gpu

MAX_ABS = 5e-3
REL_L2 = 3e-3


def _close(got, ref):
    d = got - ref
    mx = float(np.max(np.abs(d)))
    rl2 = float(np.linalg.norm(d) / max(np.linalg.norm(ref), 1e-30))
    return mx <= MAX_ABS and rl2 <= REL_L2, mx, rl2


def test_noalloc_entry_point_matches_workspace_entry_point():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import bit_kv_cache_split_gb300 as pkg
    from bit_kv_cache_split_gb300 import _binding

    pkg.build.build()
    lib = _binding.load()
    assert lib.lbkv_noalloc_scratch_bytes() == 16 << 20

    wl = inputs.Workload("noalloc", 3, 16, 4, [700, 129, 2000], bits=2, group=128, seed=41)
    t = inputs.generate(wl, "cuda")
    ref = pkg.decode_attn(t["q"], t["k_codes"], t["k_scale"], t["k_off"], t["v_codes"], t["v_scale"], t["v_off"],
                          t["seq_lens"], bits=2, group=128)
    torch.cuda.synchronize()
    ref = ref.float().cpu().numpy().astype(np.float64)

    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    outs = []
    for _ in range(2):
        out = torch.full_like(t["q"], float("nan"))
        d = _binding.make_desc(wl.batch, wl.num_q_heads, wl.num_kv_heads, wl.t_cap)
        ptrs = [ctypes.c_void_p(t[k].data_ptr()) for k in
                ("q", "k_codes", "k_scale", "k_off", "v_codes", "v_scale", "v_off", "seq_lens")]
        st = lib.lbkv_decode_attn_noalloc(ctypes.byref(d), *ptrs, 2, 0, 0, 128, ctypes.c_void_p(out.data_ptr()),
                                          stream)
        assert st == 0, _binding.strerror(st)
        torch.cuda.synchronize()
        got = out.float().cpu().numpy().astype(np.float64)
        ok, mx, rl2 = _close(got, ref)
        assert ok, f"max-abs {mx:.3e}, rel-L2 {rl2:.3e}"
        outs.append(got)
    ok, mx, rl2 = _close(outs[1], outs[0])
    assert ok, f"second call: max-abs {mx:.3e}, rel-L2 {rl2:.3e}"


def test_noalloc_rejects_scratch_beyond_the_array():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from bit_kv_cache_split_gb300 import _binding

    lib = _binding.load()
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
