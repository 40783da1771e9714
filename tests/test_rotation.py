"""Rotation folded into Q: an accuracy recipe for 2-bit caches (OSCAR's rotations, named in the
accuracy paragraph of the explainer "FOSCAR speeds up 2-bit KV decode -- Affine folding of KV
dequantization"; the related explainer "KVarN -- Hadamard-rotated 2-bit KV cache").

The stored key and/or value rows are rotated by the normalized Hadamard matrix H of order
head_dim before they are quantized. H is symmetric and orthogonal, so attention over rotated
keys takes the query rotated once by H, and the output over rotated values is rotated back once
by H: the cache is read exactly as before.

CPU tests pin the oracle's rotation: H against the Sylvester construction, orthogonality, the
fp32 butterflies against exact integer sums and the fp64 product, the bf16 rounding, the decode
definition against unrotated attention, and the accuracy gain on outlier channels."""

import numpy as np
import pytest

import oracle

D = 128


def sylvester(n):
    h = np.ones((1, 1))
    while h.shape[0] < n:
        h = np.block([[h, h], [h, -h]])
    return h / np.sqrt(n)


def bf16_bits(x):
    """Round float64 values to bf16 bit patterns (through float32, nearest-even at each step)."""
    f = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    return ((f + 0x7FFF + ((f >> 16) & 1)) >> 16).astype(np.uint16)


def bf16_value(bits):
    return (np.asarray(bits, dtype=np.uint32) << 16).view(np.float32).astype(np.float64)


@pytest.mark.parametrize("n", [1, 2, 4, 8, 16, 32, 64, 128])
def test_hadamard_matches_sylvester_construction(n):
    assert np.array_equal(oracle.hadamard(n), sylvester(n))


def test_hadamard_is_symmetric_and_orthogonal():
    H = oracle.hadamard(D)
    assert np.array_equal(H, H.T)
    assert np.abs(H @ H - np.eye(D)).max() < 1e-12
    # the first row is the constant vector, every other row sums to zero
    assert np.allclose(H.sum(axis=1), np.r_[np.sqrt(D), np.zeros(D - 1)])


@pytest.mark.parametrize("n", [0, 3, 96])
def test_hadamard_rejects_other_orders(n):
    with pytest.raises(ValueError):
        oracle.hadamard(n)


def test_rotated_rows_are_exact_on_small_integers():
    """Integers up to 255 keep every butterfly sum exact in fp32: the result is then the exact
    unnormalized Hadamard sum times fp32(1/sqrt(128)), rounded once."""
    rng = np.random.default_rng(1)
    xi = rng.integers(-255, 256, size=(16, D))
    y32, _ = oracle.rotate_rows(bf16_bits(xi))
    exact = (sylvester(D) * np.sqrt(D)).round().astype(np.int64) @ xi.T
    c = np.float32(1.0 / np.sqrt(D))
    assert np.array_equal(y32, (exact.T.astype(np.float32) * c).astype(np.float32))


def test_rotated_rows_follow_the_matrix_product():
    rng = np.random.default_rng(2)
    xb = bf16_bits(rng.normal(size=(64, D)) * np.exp(rng.normal(size=(64, 1))))
    x = bf16_value(xb)
    y32, _ = oracle.rotate_rows(xb)
    ref = x @ sylvester(D).T
    # 7 butterfly stages and the scaling, each rounded to fp32: |error| <= 8 * 2^-24 * sum|x| / sqrt(D)
    bound = 8 * 2.0 ** -24 * np.abs(x).sum(axis=1, keepdims=True) / np.sqrt(D)
    assert np.all(np.abs(y32 - ref) <= bound)


def test_rotated_rows_round_to_the_nearest_bf16():
    rng = np.random.default_rng(3)
    y32, y16 = oracle.rotate_rows(bf16_bits(rng.normal(size=(32, D))))
    lo = (y32.view(np.uint32) >> 16).astype(np.uint16)  # truncation toward zero in magnitude
    hi = lo + 1
    dlo = np.abs(bf16_value(lo) - y32)
    dhi = np.abs(bf16_value(hi) - y32)
    want = np.where(dlo < dhi, lo, np.where(dhi < dlo, hi, np.where(lo % 2 == 0, lo, hi)))
    assert np.array_equal(y16, want)


def test_rotating_twice_returns_the_row():
    rng = np.random.default_rng(4)
    xb = bf16_bits(rng.normal(size=(16, D)))
    _, y = oracle.rotate_rows(xb)
    z32, _ = oracle.rotate_rows(y)
    x = bf16_value(xb)
    # the one bf16 rounding of the first rotation, carried through an orthogonal map
    err = np.linalg.norm(z32 - x, axis=1)
    assert np.all(err <= 2.0 ** -8 * np.linalg.norm(x, axis=1) * 1.01)


def _window_problem(K, V, q_bits, rotation=0):
    """Decode inputs with no quantized tokens: the bf16 rows K, V [B][Hkv][W][D] are the window."""
    B, Hkv, W, _ = K.shape
    z8 = np.zeros((B, Hkv, 128, D // 4), np.uint8)
    z16 = np.zeros((B, Hkv, 128, 1), np.uint16)
    return oracle.DecodeInputs(q=q_bits, k_codes=z8, k_scale=z16, k_off=z16, v_codes=z8, v_scale=z16, v_off=z16,
                               seq_lens=np.zeros(B, np.int32), bits=2, k_layout=0, v_layout=0, group=128, Hkv=Hkv,
                               T_cap=128, k_win=K, v_win=V, win_lens=np.full(B, W, np.int32), win_cap=W,
                               rotation=rotation)


@pytest.mark.parametrize("rotation", [1, 2, 3])
def test_decode_over_rotated_rows_equals_attention_over_the_rows(rotation):
    """Rows stored rotated, read with the matching rotation flags, give the attention of the
    unrotated rows up to the bf16 rounding of the stored rotated rows."""
    rng = np.random.default_rng(5 + rotation)
    B, Hkv, hq, W = 2, 2, 4, 96
    K = bf16_bits(rng.normal(size=(B, Hkv, W, D)))
    V = bf16_bits(rng.normal(size=(B, Hkv, W, D)))
    q = bf16_bits(rng.normal(size=(B, Hkv * hq, D)))
    Kr = oracle.rotate_rows(K)[1] if rotation & 1 else K
    Vr = oracle.rotate_rows(V)[1] if rotation & 2 else V
    ref = oracle.decode_ref(_window_problem(K, V, q))
    got = oracle.decode_ref(_window_problem(Kr, Vr, q, rotation))
    # The stored rotated rows carry one bf16 rounding each: |dk_j| <= 2^-9 |(Hk)_j|. A score moves
    # by at most sigma sum_j |(Hq)_j| 2^-9 |(Hk)_j| =: ds, the weights by a factor within
    # e^(+-2 ds), so the output by (e^(2 ds) - 1) max|v|; rotated values add 2^-9 max |v|_2.
    H = sylvester(D)
    qh = np.abs(bf16_value(q) @ H).reshape(B, Hkv, hq, D)
    kh = np.abs(bf16_value(K) @ H)
    ds = (rotation & 1) * (np.einsum("bkid,bktd->bkit", qh, kh) * 2.0 ** -9 / np.sqrt(D)).max()
    vmax = np.abs(bf16_value(V)).max()
    dv = (rotation >> 1) * 2.0 ** -9 * np.linalg.norm(bf16_value(V), axis=-1).max()
    bound = np.expm1(2 * ds) * vmax + dv
    assert np.abs(got - ref).max() <= bound
    # a decode that ignored the rotation is far off, by two orders of magnitude more
    wrong = oracle.decode_ref(_window_problem(Kr, Vr, q, 0))
    assert np.abs(wrong - ref).max() > 100 * np.abs(got - ref).max()
    assert np.linalg.norm(wrong - ref) > 0.5 * np.linalg.norm(ref)


def test_rotation_flags_are_validated():
    rng = np.random.default_rng(9)
    K = bf16_bits(rng.normal(size=(1, 1, 8, D)))
    q = bf16_bits(rng.normal(size=(1, 1, D)))
    with pytest.raises(ValueError):
        oracle.decode_ref(_window_problem(K, K, q, 4))
    with pytest.raises(ValueError):
        oracle.decode_folded(_window_problem(K, K, q, 1))


def _int2_error(K, V, q, L, rotation):
    """rel-L2 error of INT2 token-wise g128 decode (oracle) against exact attention."""
    B, Hkv = K.shape[:2]
    lens = np.full(B, L, np.int32)
    Ks = oracle.rotate_rows(K)[1] if rotation & 1 else K
    Vs = oracle.rotate_rows(V)[1] if rotation & 2 else V
    kc, ks, kz = oracle.pack(Ks, lens, 2, 0, 128)
    vc, vs, vz = oracle.pack(Vs, lens, 2, 0, 128)
    x = oracle.DecodeInputs(q=q, k_codes=kc, k_scale=ks, k_off=kz, v_codes=vc, v_scale=vs, v_off=vz, seq_lens=lens,
                            bits=2, k_layout=0, v_layout=0, group=128, Hkv=Hkv, T_cap=K.shape[2], rotation=rotation)
    got = oracle.decode_ref(x)
    ref = oracle.decode_ref(_window_problem(K, V, q))
    return np.linalg.norm(got - ref) / np.linalg.norm(ref)


def test_rotation_lowers_int2_error_on_outlier_channels():
    """Keys with a few large channels (the case rotations are for): the rotated INT2 cache gives
    a clearly smaller decode error than the plain one."""
    rng = np.random.default_rng(10)
    B, Hkv, hq, T = 2, 2, 4, 128
    k = rng.normal(size=(B, Hkv, T, D))
    k[..., [3, 77]] *= 12.0  # outlier channels
    v = rng.normal(size=(B, Hkv, T, D))
    v[..., 40] *= 8.0
    K, V = bf16_bits(k), bf16_bits(v)
    q = bf16_bits(rng.normal(size=(B, Hkv * hq, D)) * 0.3)
    plain = _int2_error(K, V, q, T, 0)
    rotated = _int2_error(K, V, q, T, 3)
    assert rotated < 0.7 * plain, (plain, rotated)
