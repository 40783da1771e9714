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


# ------------------------------------------------------------------ GPU

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def lbkv():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import bit_kv_cache_split_gb300 as m

    m.build.build()
    m.load()
    oracle.build()
    return m


def _bf16_tensor(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)


def _bits(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


@pytest.mark.gpu
@pytest.mark.parametrize("rows", [1, 37, 4096])
def test_rotate_kernel_equals_the_oracle_bit_for_bit(lbkv, rows):
    rng = np.random.default_rng(rows)
    x = bf16_bits(rng.normal(size=(rows, D)) * np.exp(2 * rng.normal(size=(rows, 1))))
    xt = _bf16_tensor(x).cuda()
    y = lbkv.rotate(xt)
    torch.cuda.synchronize()
    assert np.array_equal(_bits(y), oracle.rotate_rows(x)[1])
    lbkv.rotate(xt, out=xt)  # in place
    torch.cuda.synchronize()
    assert np.array_equal(_bits(xt), oracle.rotate_rows(x)[1])


@pytest.mark.gpu
def test_rotate_kernel_special_values(lbkv):
    x = np.zeros((4, D), np.uint16)
    x[1, 5] = 0x7F80  # +inf
    x[2, :] = 0x8000  # -0
    x[3, 0] = 0x0001  # the smallest bf16 subnormal
    y = lbkv.rotate(_bf16_tensor(x).cuda())
    torch.cuda.synchronize()
    assert np.array_equal(_bits(y), oracle.rotate_rows(x)[1])


def _rot_wl(bits, kl, vl, g=128, hq=4, lens=(300, 1000, 129), window=0, seed=20):
    from bit_kv_cache_split_gb300 import inputs

    s = (0.01, 0.1) if bits == 2 else (0.002, 0.02)
    return inputs.Workload(f"rot-b{bits}-k{kl}-v{vl}-g{g}-hq{hq}", len(lens), 2 * hq, 2, list(lens), bits=bits,
                           k_layout=kl, v_layout=vl, group=g, s_range=s, window=window, seed=seed)


def _check_rotated_decode(m, wl, rotation, **kw):
    from bit_kv_cache_split_gb300 import inputs
    from tests.test_decode_gpu import assert_parity, run_gpu

    t = inputs.generate(wl, "cpu")
    got = run_gpu(m, t, wl, rotation=rotation, **kw)
    ref = oracle.decode_ref(oracle.inputs_from_tensors(t, bits=wl.bits, k_layout=wl.k_layout, v_layout=wl.v_layout,
                                                       group=wl.group, Hkv=wl.num_kv_heads, T_cap=wl.t_cap,
                                                       rotation=rotation))
    return assert_parity(got, ref, f"{wl.name} rotation {rotation}")


@pytest.mark.gpu
@pytest.mark.parametrize("bits", [2, 4])
@pytest.mark.parametrize("kl,vl", [(0, 0), (1, 0), (0, 1), (1, 1)])
@pytest.mark.parametrize("rotation", [1, 2, 3])
def test_rotated_decode_matches_oracle(lbkv, bits, kl, vl, rotation):
    _check_rotated_decode(lbkv, _rot_wl(bits, kl, vl), rotation)


@pytest.mark.gpu
@pytest.mark.parametrize("g,hq", [(32, 8), (64, 2), (32, 1)])
def test_rotated_decode_groups_and_gqa(lbkv, g, hq):
    _check_rotated_decode(lbkv, _rot_wl(2, 0, 0, g=g, hq=hq), 3)


@pytest.mark.gpu
def test_rotated_decode_with_window_and_empty_sequences(lbkv):
    """Window rows are stored rotated too; sequences with no cached tokens go through the
    window alone."""
    _check_rotated_decode(lbkv, _rot_wl(2, 1, 0, lens=(0, 700, 0, 33), window=50), 3)
    _check_rotated_decode(lbkv, _rot_wl(4, 0, 1, lens=(0, 129), window=7), 2)


@pytest.mark.gpu
def test_rotated_decode_single_split_and_many_splits(lbkv):
    # batch 1 with a long sequence: many CTAs merge one pair; short sequences: one CTA each
    _check_rotated_decode(lbkv, _rot_wl(2, 0, 0, lens=(20000,)), 3)
    _check_rotated_decode(lbkv, _rot_wl(2, 0, 0, lens=tuple([64] * 40)), 3)


@pytest.mark.gpu
@pytest.mark.parametrize("kl,vl", [(0, 0), (1, 0), (0, 1), (1, 1)])
def test_rotated_decode_two_level_clusters(lbkv, kl, vl):
    """Batch 1, 2 KV heads, 131,000 cached tokens and a window: on a 152-SM GPU each pair runs as
    several thread-block clusters whose partials the pair's last cluster merges with the
    window's (and rotates back)."""
    _check_rotated_decode(lbkv, _rot_wl(2, kl, vl, lens=(131000,), window=100), 3)


@pytest.mark.gpu
def test_two_level_clusters_paged_equals_contiguous(lbkv):
    from bit_kv_cache_split_gb300 import inputs

    wl = _rot_wl(2, 0, 0, lens=(131000,), window=0)
    t = inputs.generate(wl, "cpu")
    dev = {k: v.cuda() for k, v in t.items()}
    keys = ("k_codes", "k_scale", "k_off", "v_codes", "v_scale", "v_off")
    ref = lbkv.decode_attn(dev["q"], *[dev[k] for k in keys], dev["seq_lens"], bits=2, group=128)
    table, n = inputs.page_table(wl.lens, 256, wl.t_cap // 256, seed=4)
    pool = [inputs.to_pages(dev[k], table, n, 256) for k in keys]
    got = lbkv.decode_attn(dev["q"], *pool, dev["seq_lens"], bits=2, group=128, page_table=table.cuda(),
                           max_seq_len=wl.t_cap)
    torch.cuda.synchronize()
    assert torch.equal(got.view(torch.int16), ref.view(torch.int16))


@pytest.mark.gpu
def test_rotated_paged_decode_equals_rotated_contiguous(lbkv):
    from bit_kv_cache_split_gb300 import inputs

    wl = _rot_wl(2, 0, 0, lens=(300, 1000, 129))
    t = inputs.generate(wl, "cpu")
    dev = {k: v.cuda() for k, v in t.items()}
    keys = ("k_codes", "k_scale", "k_off", "v_codes", "v_scale", "v_off")
    ref = lbkv.decode_attn(dev["q"], *[dev[k] for k in keys], dev["seq_lens"], bits=2, group=128, rotation=3)
    table, n = inputs.page_table(wl.lens, 128, wl.t_cap // 128, seed=3)
    pool = [inputs.to_pages(dev[k], table, n, 128) for k in keys]
    got = lbkv.decode_attn(dev["q"], *pool, dev["seq_lens"], bits=2, group=128, rotation=3,
                           page_table=table.cuda(), max_seq_len=wl.t_cap)
    torch.cuda.synchronize()
    assert torch.equal(got.view(torch.int16), ref.view(torch.int16))


def _exact_attention(q, K, V, lens):
    """fp64 softmax attention of bf16 q [B][Hq][D] over bf16 rows K, V [B][Hkv][T][D]."""
    qf, Kf, Vf = bf16_value(q), bf16_value(K), bf16_value(V)
    B, Hq, _ = qf.shape
    hq = Hq // K.shape[1]
    out = np.zeros_like(qf)
    for b in range(B):
        for h in range(Hq):
            k, v = Kf[b, h // hq, :lens[b]], Vf[b, h // hq, :lens[b]]
            s = k @ qf[b, h] / np.sqrt(D)
            p = np.exp(s - s.max())
            out[b, h] = p @ v / p.sum()
    return out


@pytest.mark.gpu
def test_rotated_pipeline_lowers_int2_error_on_outlier_channels(lbkv):
    """rotate -> pack -> decode on the GPU, against the plain INT2 pipeline, on keys and values
    with outlier channels: the rotated pipeline equals its oracle and is clearly more accurate."""
    rng = np.random.default_rng(30)
    B, Hkv, hq, T = 4, 2, 4, 1024
    k = rng.normal(size=(B, Hkv, T, D))
    k[..., [3, 77, 100]] *= 12.0
    v = rng.normal(size=(B, Hkv, T, D))
    v[..., 40] *= 8.0
    K, V = bf16_bits(k), bf16_bits(v)
    q = bf16_bits(rng.normal(size=(B, Hkv * hq, D)) * 0.3)
    lens = [1024, 700, 1, 333]
    exact = _exact_attention(q, K, V, lens)
    sl = torch.tensor(lens, dtype=torch.int32).cuda()
    qt = _bf16_tensor(q).cuda()
    errs = {}
    for rotation in (0, 3):
        Kt, Vt = _bf16_tensor(K).cuda(), _bf16_tensor(V).cuda()
        if rotation:
            Kt, Vt = lbkv.rotate(Kt), lbkv.rotate(Vt)
        kc = lbkv.pack(Kt, sl, bits=2, layout=0, group=128)
        vc = lbkv.pack(Vt, sl, bits=2, layout=0, group=128)
        out = lbkv.decode_attn(qt, *kc, *vc, sl, bits=2, group=128, rotation=rotation)
        torch.cuda.synchronize()
        got = out.float().cpu().numpy().astype(np.float64)
        errs[rotation] = np.linalg.norm(got - exact) / np.linalg.norm(exact)
        # the GPU pipeline against the oracle's own: rotate, pack, decode
        Ks = oracle.rotate_rows(K)[1] if rotation else K
        Vs = oracle.rotate_rows(V)[1] if rotation else V
        lens_np = np.asarray(lens, np.int32)
        okc, oks, okz = oracle.pack(Ks, lens_np, 2, 0, 128)
        ovc, ovs, ovz = oracle.pack(Vs, lens_np, 2, 0, 128)
        for got_side, want_side in ((kc, (okc, oks, okz)), (vc, (ovc, ovs, ovz))):  # bit for bit
            assert np.array_equal(got_side[0].cpu().numpy(), want_side[0])
            assert np.array_equal(_bits(got_side[1]), want_side[1]) and np.array_equal(_bits(got_side[2]), want_side[2])
        ref = oracle.decode_ref(oracle.DecodeInputs(q=q, k_codes=okc, k_scale=oks, k_off=okz, v_codes=ovc,
                                                    v_scale=ovs, v_off=ovz, seq_lens=lens_np, bits=2, k_layout=0,
                                                    v_layout=0, group=128, Hkv=Hkv, T_cap=T, rotation=rotation))
        # Outputs here reach ~20 (a value row with an outlier channel, e.g. the one-token
        # sequence), where half a bf16 ulp of the output alone is up to 2^-8 |ref|: the decode
        # bar's 5e-3 holds on top of that rounding, and rel-L2 as it stands.
        from tests.test_decode_gpu import MAX_ABS, REL_L2

        assert np.all(np.abs(got - ref) <= 2.0 ** -8 * np.abs(ref) + MAX_ABS), f"pipeline rotation {rotation}"
        assert np.linalg.norm(got - ref) <= REL_L2 * np.linalg.norm(ref)
    assert errs[3] < 0.7 * errs[0], errs


@pytest.mark.gpu
@pytest.mark.parametrize("bits", [2, 4])
@pytest.mark.parametrize("kl,vl,rotation", [(0, 0, 3), (0, 0, 1), (1, 0, 3), (0, 1, 2), (1, 1, 3)])
def test_rotated_append_equals_packing_the_rotated_history(lbkv, bits, kl, vl, rotation):
    B, Hkv, T, g = 2, 2, 512, 128
    lens0 = [0, 128]
    n = g + 5
    gen = torch.Generator().manual_seed(40)
    xk = torch.randn((B, Hkv, T, D), generator=gen).to(torch.bfloat16)
    xv = torch.randn((B, Hkv, T, D), generator=gen).to(torch.bfloat16)
    hk = oracle.rotate_rows(_bits(xk))[1] if rotation & 1 else _bits(xk)
    hv = oracle.rotate_rows(_bits(xv))[1] if rotation & 2 else _bits(xv)
    l0 = torch.tensor(lens0, dtype=torch.int32).cuda()
    # the first lens0 tokens packed from the rotated history, the rest appended one by one
    k = lbkv.pack(_bf16_tensor(hk).cuda(), l0, bits=bits, layout=kl, group=g)
    v = lbkv.pack(_bf16_tensor(hv).cuda(), l0, bits=bits, layout=vl, group=g)
    windowed = kl == 1 or vl == 1
    win = {}
    if windowed:
        win = dict(k_win=torch.zeros((B, Hkv, 128, D), dtype=torch.bfloat16, device="cuda"),
                   v_win=torch.zeros((B, Hkv, 128, D), dtype=torch.bfloat16, device="cuda"),
                   win_lens=torch.zeros((B,), dtype=torch.int32, device="cuda"))
    lens = l0.clone()
    xkd, xvd = xk.cuda(), xv.cuda()
    for step in range(n):
        pos = [L + step for L in lens0]
        kn = torch.stack([xkd[b, :, p] for b, p in enumerate(pos)]).contiguous()
        vn = torch.stack([xvd[b, :, p] for b, p in enumerate(pos)]).contiguous()
        lbkv.append(kn, vn, lens, *k, *v, bits=bits, k_layout=kl, v_layout=vl, group=g, rotation=rotation, **win)
    torch.cuda.synchronize()
    final = [L + (g if windowed else n) for L in lens0]
    assert lens.cpu().tolist() == final
    for (c, s, z), h, layout in ((k, hk, kl), (v, hv, vl)):
        rc, rs, rz = oracle.pack(h, np.asarray(final, np.int32), bits, layout, g)
        for b, L in enumerate(final):
            m = L if layout == 0 else (L + g - 1) // g
            assert np.array_equal(c[b, :, :L].cpu().numpy(), rc[b, :, :L]), ("codes", b)
            assert np.array_equal(_bits(s[b, :, :m]), rs[b, :, :m]), ("scale", b)
            assert np.array_equal(_bits(z[b, :, :m]), rz[b, :, :m]), ("offset", b)
    if windowed:  # the window holds the last 5 tokens, rotated as stored
        for w, h in ((win["k_win"], hk), (win["v_win"], hv)):
            for b, L in enumerate(final):
                assert np.array_equal(_bits(w[b, :, :5]), h[b, :, L:L + 5])


@pytest.mark.gpu
@pytest.mark.parametrize("kl,vl", [(0, 0), (1, 0)])
def test_rotated_paged_append_then_decode(lbkv, kl, vl):
    """Rotation, paging and append together: a paged cache grown by rotated appends holds the
    oracle's packing of the rotated history, and decodes like its contiguous gather."""
    from bit_kv_cache_split_gb300 import inputs

    B, Hkv, T, P, g, bits = 2, 2, 512, 256, 128, 2
    lens0 = [0, 256]
    n = g + 3
    gen = torch.Generator().manual_seed(50)
    xk = torch.randn((B, Hkv, T, D), generator=gen).to(torch.bfloat16)
    xv = torch.randn((B, Hkv, T, D), generator=gen).to(torch.bfloat16)
    hk, hv = oracle.rotate_rows(_bits(xk))[1], oracle.rotate_rows(_bits(xv))[1]
    table, num_pages = inputs.page_table([T] * B, P, T // P, seed=51)
    tab = table.cuda()
    l0 = torch.tensor(lens0, dtype=torch.int32).cuda()
    paged = dict(page_table=tab, num_pages=num_pages, page_tokens=P)
    k = lbkv.pack(lbkv.rotate(xk.cuda()), l0, bits=bits, layout=kl, group=g, **paged)
    v = lbkv.pack(lbkv.rotate(xv.cuda()), l0, bits=bits, layout=vl, group=g, **paged)
    windowed = kl == 1 or vl == 1
    win = {}
    if windowed:
        win = dict(k_win=torch.zeros((B, Hkv, 128, D), dtype=torch.bfloat16, device="cuda"),
                   v_win=torch.zeros((B, Hkv, 128, D), dtype=torch.bfloat16, device="cuda"),
                   win_lens=torch.zeros((B,), dtype=torch.int32, device="cuda"))
    lens = l0.clone()
    xkd, xvd = xk.cuda(), xv.cuda()
    for step in range(n):
        pos = [L + step for L in lens0]
        kn = torch.stack([xkd[b, :, p] for b, p in enumerate(pos)]).contiguous()
        vn = torch.stack([xvd[b, :, p] for b, p in enumerate(pos)]).contiguous()
        lbkv.append(kn, vn, lens, *k, *v, bits=bits, k_layout=kl, v_layout=vl, group=g, rotation=3, page_table=tab,
                    max_seq_len=T, **win)
    torch.cuda.synchronize()
    final = [L + (g if windowed else n) for L in lens0]
    assert lens.cpu().tolist() == final
    for (c, s, z), h, layout in ((k, hk, kl), (v, hv, vl)):
        r = 1 if layout == 0 else g
        cc, ss, zz = (inputs.from_pages(a, table, T // rr) for a, rr in ((c, 1), (s, r), (z, r)))
        rc, rs, rz = oracle.pack(h, np.asarray(final, np.int32), bits, layout, g)
        for b, L in enumerate(final):
            m = L if layout == 0 else (L + g - 1) // g
            assert np.array_equal(cc[b, :, :L].cpu().numpy(), rc[b, :, :L]), ("codes", b)
            assert np.array_equal(_bits(ss[b, :, :m]), rs[b, :, :m]), ("scale", b)
            assert np.array_equal(_bits(zz[b, :, :m]), rz[b, :, :m]), ("offset", b)
    q = torch.randn((B, 4 * Hkv, D), generator=gen).to(torch.bfloat16).cuda()
    common = dict(bits=bits, k_layout=kl, v_layout=vl, group=g, rotation=3, **win)
    got = lbkv.decode_attn(q, *k, *v, lens, page_table=tab, max_seq_len=T, **common)
    gather = lambda side, layout: [inputs.from_pages(a, table, T // rr)  # noqa: E731
                                   for a, rr in ((side[0], 1), (side[1], 1 if layout == 0 else g),
                                                 (side[2], 1 if layout == 0 else g))]
    ref = lbkv.decode_attn(q, *gather(k, kl), *gather(v, vl), lens, **common)
    torch.cuda.synchronize()
    assert torch.equal(got.view(torch.int16), ref.view(torch.int16))
