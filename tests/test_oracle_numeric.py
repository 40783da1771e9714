"""Pins of the CPU oracle against library routines, closed forms, invariants and
the exactness of affine folding. None of these compares the oracle with a
retyped copy of itself: the references are numpy/torch routines, special cases
with a closed form, or structural invariants."""

import itertools

import numpy as np
import pytest
import torch

import oracle
from bit_kv_cache_split_gb300 import inputs
from tests.helpers import (bits16, f16_to_np, np_dequant, np_unpack, sdpa_reference, to_oracle,
                           golden_lines, bf16_to_np)


# ----------------------------------------------------------- number formats

def test_fp16_decode_all_patterns(oracle_lib):
    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = pats.view(np.float16).astype(np.float64)
    got = np.array([oracle.fp16_to_f64(int(p)) for p in pats])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def test_fp16_encode_matches_numpy_rne(oracle_lib):
    rng = np.random.default_rng(0)
    xs = np.concatenate([
        rng.standard_normal(20000).astype(np.float32) * np.float32(10.0) ** rng.integers(-8, 5, 20000).astype(np.float32),
        # exact halfway points between neighbouring fp16 values, both parities
        (np.arange(0, 2048, dtype=np.float32) + np.float32(0.5)) * np.float32(2.0 ** -24),
        (np.arange(1024, 2048, dtype=np.float32) + np.float32(0.5)) * np.float32(2.0 ** -3),
        np.array([65504, 65519.99, 65520, 70000, 5.96e-8, 2.98e-8, 2.9802322e-08, -0.0], dtype=np.float32),
    ])
    with np.errstate(over="ignore"):  # values past the fp16 range round to infinity, as they should
        ref = xs.astype(np.float16).view(np.uint16)
    got = np.array([oracle.f64_to_fp16(float(x)) for x in xs], dtype=np.uint16)
    assert np.array_equal(got, ref)


def test_bf16_decode_matches_torch(oracle_lib):
    rng = np.random.default_rng(1)
    pats = rng.integers(0, 65536, 5000).astype(np.uint16)
    pats = pats[(pats & 0x7F80) != 0x7F80]  # finite only
    ref = torch.from_numpy(pats.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    got = np.array([oracle.bf16_to_f64(int(p)) for p in pats])
    assert np.array_equal(got, ref)


def test_independent_unpack_agrees_with_golden_table():
    """The tests' own numpy unpack (used to feed library routines) follows the same bit table."""
    for line in golden_lines("unpack_bits.txt"):
        f = line.split()
        bits, byte, codes = int(f[0]), int(f[1], 16), [int(x) for x in f[2:]]
        assert np_unpack(np.array([[byte]], np.uint8), bits)[0].tolist() == codes


# ----------------------------------------------------- decode vs libraries

LAYOUTS = [(0, 0), (1, 0), (0, 1), (1, 1)]


def _small(bits, kl, vl, g, hq, lens, seed, window=0, q_std=1.0, sm_scale=0.0, hkv=2):
    s = (0.01, 0.1) if bits == 2 else (0.002, 0.02)
    return inputs.Workload("t", len(lens), hq * hkv, hkv, list(lens), bits=bits, k_layout=kl, v_layout=vl,
                           group=g, s_range=s, seed=seed, window=window, q_std=q_std, sm_scale=sm_scale)


def _dense(t, wl):
    k = np_dequant(t["k_codes"].numpy(), f16_to_np(t["k_scale"]), f16_to_np(t["k_off"]), wl.bits, wl.k_layout, wl.group)
    v = np_dequant(t["v_codes"].numpy(), f16_to_np(t["v_scale"]), f16_to_np(t["v_off"]), wl.bits, wl.v_layout, wl.group)
    return k, v


@pytest.mark.parametrize("bits", [2, 4])
@pytest.mark.parametrize("layouts", LAYOUTS)
def test_decode_ref_matches_torch_sdpa(oracle_lib, bits, layouts):
    """Dequantize-then-attend equals torch's fp64 scaled_dot_product_attention on the
    dense s*q+z cache, with GQA, ragged lengths and partial channel groups."""
    for g, hq, seed in [(128, 4, 0), (64, 2, 1), (32, 1, 2), (32, 8, 3)]:
        wl = _small(bits, *layouts, g, hq, [300, 129, 1], seed, q_std=3.0)
        t = inputs.generate(wl)
        got = oracle.decode_ref(to_oracle(t, wl))
        k, v = _dense(t, wl)
        ref = sdpa_reference(bf16_to_np(t["q"]), k, v, wl.lens, sm_scale=1 / np.sqrt(128))
        np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-13)


def test_decode_ref_integer_attention(oracle_lib):
    """b=4, g=D, token-wise, s=1, z=0: the cache holds plain integers; attention over them
    is textbook SDPA on the integer matrix (no affine step involved)."""
    rng = np.random.default_rng(7)
    B, Hkv, hq, D, T, L = 1, 2, 4, 128, 128, 97
    codes_int = rng.integers(0, 16, (B, Hkv, T, D))
    packed = (codes_int[..., 0::2] | (codes_int[..., 1::2] << 4)).astype(np.uint8)
    ones = np.full((B, Hkv, T, 1), 0x3C00, np.uint16)
    zeros = np.zeros((B, Hkv, T, 1), np.uint16)
    q = (rng.standard_normal((B, Hkv * hq, D)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    x = oracle.DecodeInputs(q=q, k_codes=packed, k_scale=ones, k_off=zeros, v_codes=packed, v_scale=ones,
                            v_off=zeros, seq_lens=[L], bits=4, k_layout=0, v_layout=0, group=D, Hkv=Hkv, T_cap=T,
                            sm_scale=0.05)
    got = oracle.decode_ref(x)
    qf = (q.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    ref = sdpa_reference(qf, codes_int.astype(np.float64), codes_int.astype(np.float64), [L], sm_scale=0.05)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)


def test_window_matches_sdpa_on_concatenation(oracle_lib):
    """The bf16 window is attended after the quantized tokens: softmax over the union."""
    wl = _small(2, 0, 0, 128, 4, [200, 0, 77], 5, window=16, q_std=2.0)
    t = inputs.generate(wl)
    t["win_lens"] = torch.tensor([16, 9, 0], dtype=torch.int32)
    got = oracle.decode_ref(to_oracle(t, wl))
    k, v = _dense(t, wl)
    kw, vw = bf16_to_np(t["k_win"]), bf16_to_np(t["v_win"])
    B, Hkv = k.shape[:2]
    out = np.zeros_like(got)
    for b in range(B):
        L, W = wl.lens[b], int(t["win_lens"][b])
        kk = np.concatenate([k[b:b + 1, :, :L], kw[b:b + 1, :, :W]], axis=2)
        vv = np.concatenate([v[b:b + 1, :, :L], vw[b:b + 1, :, :W]], axis=2)
        out[b:b + 1] = sdpa_reference(bf16_to_np(t["q"][b:b + 1]), kk, vv, [L + W], sm_scale=1 / np.sqrt(128))
    np.testing.assert_allclose(got, out, rtol=1e-12, atol=1e-13)


# ---------------------------------------------- closed forms and invariants

def test_zero_query_gives_mean_of_values(oracle_lib):
    """Q = 0: every score is equal, so the output is the plain mean of the valid V rows."""
    wl = _small(2, 0, 1, 128, 4, [257, 1000], 11)
    t = inputs.generate(wl)
    t["q"] = torch.zeros_like(t["q"])
    got = oracle.decode_ref(to_oracle(t, wl))
    _, v = _dense(t, wl)
    for b, L in enumerate(wl.lens):
        mean = v[b, :, :L].mean(axis=1)  # [Hkv][D]
        np.testing.assert_allclose(got[b], np.repeat(mean, 4, axis=0), rtol=1e-12, atol=1e-14)


def test_constant_values_weights_sum_to_one(oracle_lib):
    """s = 0 and one offset everywhere: the output equals that offset (weights sum to 1)."""
    wl = _small(4, 0, 0, 64, 2, [333], 12, q_std=4.0)
    t = inputs.generate(wl)
    t["v_scale"].zero_()
    t["v_off"].fill_(0.3125)
    got = oracle.decode_ref(to_oracle(t, wl))
    np.testing.assert_allclose(got, 0.3125, rtol=1e-15, atol=0)


def test_one_hot_score_returns_that_value_row(oracle_lib):
    """A score far above the rest puts all the weight on one token."""
    wl = _small(2, 0, 0, 128, 1, [64], 13, hkv=1)
    t = inputs.generate(wl)
    codes = np.zeros((1, 1, 128, 32), np.uint8)
    codes[0, 0, 17, :] = 0xFF  # token 17 has every code 3, the rest 0
    t["k_codes"] = torch.from_numpy(codes)
    t["k_scale"].fill_(1.0)
    t["k_off"].zero_()
    t["q"] = torch.full_like(t["q"], 1.0)
    wl.sm_scale = 1.0  # score 384 for token 17, 0 for the others
    got = oracle.decode_ref(to_oracle(t, wl))
    _, v = _dense(t, wl)
    np.testing.assert_allclose(got[0, 0], v[0, 0, 17], rtol=1e-12, atol=1e-12)


def test_gqa_head_mapping(oracle_lib):
    """Query head h reads KV head h // (Hq/Hkv): with Q = 0 and a distinct constant per KV
    head, each output row names its KV head."""
    wl = _small(2, 0, 0, 128, 4, [50], 14, hkv=3)
    t = inputs.generate(wl)
    t["q"] = torch.zeros_like(t["q"])
    t["v_scale"].zero_()
    for kv in range(3):
        t["v_off"][:, kv] = float(kv + 1)
    got = oracle.decode_ref(to_oracle(t, wl))
    for h in range(12):
        assert np.all(got[0, h] == h // 4 + 1)


def test_empty_sequence_gives_zero_row(oracle_lib):
    wl = _small(2, 0, 0, 128, 2, [0, 5], 15)
    t = inputs.generate(wl)
    got = oracle.decode_ref(to_oracle(t, wl))
    assert np.all(got[0] == 0) and np.all(np.isfinite(got))
    assert np.any(got[1] != 0)


def test_window_split_invariance(oracle_lib):
    """Moving the last tokens from the quantized cache into the bf16 window (values that
    are exact in both formats) leaves the output unchanged."""
    rng = np.random.default_rng(16)
    D, T, L, W = 128, 128, 40, 8
    ci = rng.integers(0, 4, (1, 1, T, D))
    packed = (ci[..., 0::4] | (ci[..., 1::4] << 2) | (ci[..., 2::4] << 4) | (ci[..., 3::4] << 6)).astype(np.uint8)
    one = np.full((1, 1, T, 1), 0x3C00, np.uint16)
    zero = np.zeros((1, 1, T, 1), np.uint16)
    q = (rng.standard_normal((1, 2, D)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    full = oracle.DecodeInputs(q=q, k_codes=packed, k_scale=one, k_off=zero, v_codes=packed, v_scale=one,
                               v_off=zero, seq_lens=[L], bits=2, k_layout=0, v_layout=0, group=D, Hkv=1, T_cap=T)
    win = np.zeros((1, 1, W, D), np.float32)
    win[0, 0] = ci[0, 0, L - W:L]
    winb = (win.view(np.uint32) >> 16).astype(np.uint16)
    split = oracle.DecodeInputs(q=q, k_codes=packed, k_scale=one, k_off=zero, v_codes=packed, v_scale=one,
                                v_off=zero, seq_lens=[L - W], bits=2, k_layout=0, v_layout=0, group=D, Hkv=1,
                                T_cap=T, k_win=winb, v_win=winb, win_lens=[W], win_cap=W)
    np.testing.assert_allclose(oracle.decode_ref(split), oracle.decode_ref(full), rtol=1e-14, atol=1e-15)


def test_rows_subset_and_threads_agree(oracle_lib):
    wl = _small(4, 1, 0, 128, 4, [700, 130], 17)
    t = inputs.generate(wl)
    x = to_oracle(t, wl)
    full = oracle.decode_ref(x, n_threads=1)
    rows = [(1, 7), (0, 0), (1, 3)]
    sub = oracle.decode_ref(x, rows=rows, n_threads=3)
    for i, (b, h) in enumerate(rows):
        assert np.array_equal(sub[i], full[b, h])
    assert np.array_equal(oracle.decode_ref(x, n_threads=5), full)


# ------------------------------------------------ folding is exact (fp64)

@pytest.mark.parametrize("bits", [2, 4])
@pytest.mark.parametrize("layouts", LAYOUTS)
def test_folded_equals_dequantized_attention(oracle_lib, bits, layouts):
    """The four fold formulas inside an online softmax reproduce the dequantized
    attention output to fp64 rounding, including partial groups and masking."""
    for g, hq in itertools.product([32, 64, 128], [1, 2, 4, 8]):
        wl = _small(bits, *layouts, g, hq, [300, 129, 33, 0], seed=g + hq, q_std=3.0, hkv=1)
        t = inputs.generate(wl)
        x = to_oracle(t, wl)
        ref = oracle.decode_ref(x)
        for block in (128, 256):
            got, _, _ = oracle.decode_folded(x, block=block)
            assert np.max(np.abs(got - ref)) <= 1e-12, (g, hq, block)


def test_folded_with_window_equals_reference(oracle_lib):
    wl = _small(2, 0, 1, 64, 4, [150, 7], 21, window=12, q_std=2.0)
    t = inputs.generate(wl)
    x = to_oracle(t, wl)
    got, _, _ = oracle.decode_folded(x, block=128)
    assert np.max(np.abs(got - oracle.decode_ref(x))) <= 1e-12


@pytest.mark.parametrize("k_layout", [0, 1])
def test_key_offset_after_softmax_is_wrong(oracle_lib, k_layout):
    """Negative test: the key-side offset must reach the scores before the softmax."""
    wl = _small(2, k_layout, 0, 128, 4, [384], 22, q_std=3.0, hkv=1)
    t = inputs.generate(wl)
    x = to_oracle(t, wl)
    ref = oracle.decode_ref(x)
    bad, _, _ = oracle.decode_folded(x, block=128, misorder=1)
    assert np.max(np.abs(bad - ref)) > 1e-4


def test_channelwise_key_offset_single_group_is_softmax_invariant(oracle_lib):
    """With one token group the channel-wise key offset is one constant per query and the
    softmax cancels it; the ordering rule only bites across groups (checked above)."""
    wl = _small(2, 1, 0, 128, 4, [100], 23, q_std=3.0, hkv=1)
    t = inputs.generate(wl)
    x = to_oracle(t, wl)
    bad, _, _ = oracle.decode_folded(x, block=128, misorder=1)
    assert np.max(np.abs(bad - oracle.decode_ref(x))) <= 1e-12


@pytest.mark.parametrize("v_layout", [0, 1])
def test_value_offset_after_division_is_wrong(oracle_lib, v_layout):
    """Negative test: the value-side offset must land before the division by l."""
    wl = _small(2, 0, v_layout, 128, 4, [384], 24, q_std=3.0, hkv=1)
    t = inputs.generate(wl)
    x = to_oracle(t, wl)
    bad, _, _ = oracle.decode_folded(x, block=128, misorder=2)
    assert np.max(np.abs(bad - oracle.decode_ref(x))) > 1e-3


# ------------------------------------------------------------- quantizer

def _bf16_from(x: np.ndarray) -> np.ndarray:
    return torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("bits", [2, 4])
@pytest.mark.parametrize("layout", [0, 1])
def test_pack_reconstruction_bound(oracle_lib, bits, layout):
    """Every valid value is within half a step of its reconstruction s*q + z, up to the
    fp16 rounding of s and z (brute force over random groups)."""
    rng = np.random.default_rng(30 + bits + layout)
    B, Hkv, D, g = 2, 2, 128, 64
    lens = [200, 129]
    T = 256
    x = rng.standard_normal((B, Hkv, T, D)) * rng.uniform(0.1, 3.0)
    xb = _bf16_from(x)
    xf = (xb.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    codes, s, z = oracle.pack(xb, lens, bits, layout, g)
    q = np_unpack(codes, bits)
    sv = s.view(np.float16).astype(np.float64)
    zv = z.view(np.float16).astype(np.float64)
    if layout == 0:
        S, Z = np.repeat(sv, g, -1), np.repeat(zv, g, -1)
    else:
        S, Z = np.repeat(sv, g, -2), np.repeat(zv, g, -2)
    rec = S * q + Z
    qmax = (1 << bits) - 1
    for b, L in enumerate(lens):
        err = np.abs(rec[b, :, :L] - xf[b, :, :L])
        # half a step, plus fp16 rounding of s (relative 2^-11, times at most qmax steps)
        # and of z (half an fp16 ulp of the group minimum)
        bound = S[b, :, :L] * (0.5 + qmax * 2.0 ** -10) + np.abs(Z[b, :, :L]) * 2.0 ** -10 + 1e-12
        assert np.all(err <= bound)
        assert np.all(codes[b, :, L:] == 0)


def test_pack_padding_and_partial_group(oracle_lib):
    """Padding tokens get code 0 and leave s/z untouched; the last channel-wise group sees
    only valid tokens (changing padded inputs changes nothing)."""
    rng = np.random.default_rng(40)
    B, Hkv, D, T, g, L = 1, 1, 128, 256, 128, 150
    x = rng.standard_normal((B, Hkv, T, D))
    x2 = x.copy()
    x2[:, :, L:] = 1000.0
    sentinel = np.full((B, Hkv, T // g, D), 0x1234, np.uint16)
    c1, s1, z1 = oracle.pack(_bf16_from(x), [L], 2, 1, g, scale_init=sentinel, off_init=sentinel)
    c2, s2, z2 = oracle.pack(_bf16_from(x2), [L], 2, 1, g, scale_init=sentinel, off_init=sentinel)
    assert np.array_equal(c1, c2) and np.array_equal(s1, s2) and np.array_equal(z1, z2)
    assert np.all(c1[:, :, L:] == 0)
    # token-wise: padding rows untouched
    sent_t = np.full((B, Hkv, T, 1), 0x1234, np.uint16)
    _, st, zt = oracle.pack(_bf16_from(x), [L], 2, 0, 128, scale_init=sent_t, off_init=sent_t)
    assert np.all(st[:, :, L:] == 0x1234) and np.all(zt[:, :, L:] == 0x1234)
    assert not np.any(st[:, :, :L] == 0x1234)


def test_pack_constant_group_has_zero_scale(oracle_lib):
    x = np.full((1, 1, 128, 128), 0.75)
    codes, s, z = oracle.pack(_bf16_from(x), [128], 4, 0, 32)
    assert np.all(s == 0) and np.all(codes == 0)
    assert np.all(z.view(np.float16) == np.float16(0.75))


@pytest.mark.parametrize("bits", [2, 4])
def test_pack_scale_offset_are_fp16_of_group_extremes(oracle_lib, bits):
    """z is numpy's fp16 of the group minimum and s numpy's fp16 of the single-precision
    (max - min) / (2^b - 1), bit for bit (token-wise groups of 32 channels)."""
    rng = np.random.default_rng(50 + bits)
    x = rng.standard_normal((1, 2, 128, 128)) * 7.0
    xb = _bf16_from(x)
    xf = (xb.astype(np.uint32) << 16).view(np.float32)
    _, s, z = oracle.pack(xb, [128], bits, 0, 32)
    grp = xf.reshape(1, 2, 128, 4, 32)
    mn, mx = grp.min(-1), grp.max(-1)
    step = (mx - mn) / np.float32((1 << bits) - 1)
    assert step.dtype == np.float32
    assert np.array_equal(z, mn.astype(np.float16).view(np.uint16))
    assert np.array_equal(s, step.astype(np.float16).view(np.uint16))


def test_pack_signed_zero_extremes_read_as_positive_zero(oracle_lib):
    """A group whose minimum (or maximum) is -0 stores z = +0 and s = +0 (this library's
    reading of the quantizer: scale and offset never carry a negative zero)."""
    x = np.zeros((1, 1, 128, 128), np.float32)
    x[0, 0, :, ::2] = -0.0
    codes, s, z = oracle.pack(_bf16_from(x), [128], 2, 0, 32)
    assert np.all(s == 0) and np.all(z == 0) and np.all(codes == 0)
