"""The BF16 comparator: its oracle (plain softmax attention over a bf16 cache, through the
decode definition's window step) pinned to closed forms, the C ABI's argument checks, and
the CUDA kernels against the oracle."""

import ctypes

import numpy as np
import pytest
import torch

import oracle
from tests.helpers import bits16


def _bf16(x):
    return bits16(torch.from_numpy(np.asarray(x, np.float32)).to(torch.bfloat16))


def test_oracle_equal_scores_give_the_mean(oracle_lib):
    """Q = 0: every token has the same score, the output is the mean of V over the valid tokens."""
    rng = np.random.default_rng(1)
    B, Hkv, hq, T, D = 2, 2, 3, 40, 128
    k = rng.standard_normal((B, Hkv, T, D))
    v = rng.standard_normal((B, Hkv, T, D))
    q = np.zeros((B, Hkv * hq, D))
    lens = [40, 7]
    out = oracle.attention_bf16(_bf16(q), _bf16(k), _bf16(v), lens)
    vb = torch.from_numpy(v.astype(np.float32)).to(torch.bfloat16).double().numpy()
    for b, L in enumerate(lens):
        for h in range(Hkv * hq):
            np.testing.assert_allclose(out[b, h], vb[b, h // hq, :L].mean(axis=0), rtol=1e-12, atol=1e-14)


def test_oracle_one_hot_score_returns_that_row(oracle_lib):
    B, Hkv, T, D = 1, 1, 16, 128
    k = np.zeros((B, Hkv, T, D))
    k[0, 0, 5, 0] = 64.0
    v = np.random.default_rng(2).standard_normal((B, Hkv, T, D))
    q = np.zeros((B, 1, D))
    q[0, 0, 0] = 64.0  # score 4096 / sqrt(128) on token 5, 0 elsewhere
    out = oracle.attention_bf16(_bf16(q), _bf16(k), _bf16(v), [T])
    vb = torch.from_numpy(v.astype(np.float32)).to(torch.bfloat16).double().numpy()
    np.testing.assert_allclose(out[0, 0], vb[0, 0, 5], rtol=0, atol=1e-12)


def test_oracle_empty_sequence_is_zero(oracle_lib):
    k = np.ones((1, 1, 8, 128))
    out = oracle.attention_bf16(_bf16(np.ones((1, 4, 128))), _bf16(k), _bf16(k), [0])
    assert np.all(out == 0.0)


@pytest.fixture(scope="module")
def lib():
    from bit_kv_cache_split_gb300 import _binding, build

    build.build()
    return _binding.load()


def _desc(B=1, Hq=32, Hkv=8, T=4096, D=128):
    from bit_kv_cache_split_gb300 import _binding

    return _binding.make_desc(B, Hq, Hkv, T, D)


@pytest.mark.parametrize("kw,want", [(dict(D=64), -3), (dict(Hq=30), -1), (dict(Hq=80, Hkv=8), -3), (dict(T=1000), -1),
                                     (dict(B=-1), -1)])
def test_bf16_invalid_arguments(lib, kw, want):
    d = _desc(**kw)
    null = ctypes.c_void_p(0)
    assert lib.lbkv_decode_bf16(ctypes.byref(d), *([null] * 5), null) == want
    assert lib.lbkv_bf16_workspace_bytes(ctypes.byref(d)) == 0


def test_bf16_rules(lib):
    d = _desc()
    assert lib.lbkv_bf16_workspace_bytes(ctypes.byref(d)) > 0
    null = ctypes.c_void_p(0)
    assert lib.lbkv_decode_bf16(ctypes.byref(d), *([null] * 5), null) == -1  # null pointers
    d.k_win = d.v_win = d.win_lens = 4096
    d.win_cap = 16
    assert lib.lbkv_decode_bf16(ctypes.byref(d), *([null] * 5), null) == -3  # no window
    assert lib.lbkv_decode_bf16(None, *([null] * 5), null) == -1
    e = _desc(B=0)
    assert lib.lbkv_decode_bf16(ctypes.byref(e), *([null] * 5), null) == 0


# ---------------------------------------------------------------- GPU parity

# The comparator's bound follows from its arithmetic: a bf16 output rounds by up to half an
# ulp (2^-8 relative), bf16 softmax weights by 2^-9 relative each (at most 2^-9 max|V| on
# the weighted sum), plus fp32 accumulation and exp2 approximation (well under 1e-3).
REL_L2 = 3e-3


def _bound(ref, vmax):
    return 2.0 ** -8 * np.abs(ref) + 2.0 ** -9 * vmax + 1e-3


def _run(hq, lens, T, seed, sm_scale=0.0):
    import bit_kv_cache_split_gb300 as m

    B, Hkv, D = len(lens), 2, 128
    g = torch.Generator().manual_seed(seed)
    q = torch.randn((B, Hkv * hq, D), generator=g).to(torch.bfloat16)
    k = torch.randn((B, Hkv, T, D), generator=g).to(torch.bfloat16)
    v = torch.randn((B, Hkv, T, D), generator=g).to(torch.bfloat16)
    lt = torch.tensor(lens, dtype=torch.int32)
    out = m.decode_bf16(q.cuda(), k.cuda(), v.cuda(), lt.cuda(), sm_scale=sm_scale)
    torch.cuda.synchronize()
    ref = oracle.attention_bf16(bits16(q), bits16(k), bits16(v), lens, sm_scale=sm_scale)
    got = out.float().cpu().numpy().astype(np.float64)
    d = got - ref
    vmax = float(v.float().abs().max())
    excess = float(np.max(np.abs(d) - _bound(ref, vmax)))
    rl2 = float(np.linalg.norm(d) / max(np.linalg.norm(ref), 1e-30))
    assert np.all(np.isfinite(got))
    assert excess <= 0.0 and rl2 <= REL_L2, (hq, lens, excess, rl2)


@pytest.mark.gpu
@pytest.mark.parametrize("hq", [1, 2, 4, 8])
def test_bf16_matches_oracle(hq):
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    _run(hq, [0, 1, 63, 700, 1535], 1536, seed=hq)


@pytest.mark.gpu
def test_bf16_long_and_scaled():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    _run(4, [32768, 4097], 32768, seed=9)
    _run(4, [300, 129], 384, seed=10, sm_scale=0.3)
