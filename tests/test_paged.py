"""Paged KV cache: the codes, scales and offsets live in pools of fixed-size pages that a
per-sequence page table names, as serving engines keep their caches (the SGLang
integration in the abstract of "FOSCAR: Accelerating Decode Attention over 2- and 4-Bit
KV Caches through Affine Folding").

Paging changes where a token is stored, never what is computed: a paged decode equals
the contiguous decode of the same cache bit for bit, and a paged pack or append stores
exactly the rows that the contiguous path stores. Entries outside the pool are reported
through the device status word (5) and read as page 0, never out of bounds."""

import ctypes

import numpy as np
import pytest
import torch

import oracle
from bit_kv_cache_split_gb300 import inputs
from tests.helpers import bits16
from tests.test_abi import _desc, lib  # noqa: F401  (fixture)

D = 128


# ------------------------------------------------------------------ host side (CPU)

def test_page_table_gives_each_page_one_owner():
    lens = [300, 0, 513, 128, 1]
    t, n = inputs.page_table(lens, 128, 6, spare_pages=4, seed=9)
    used = t[t >= 0].tolist()
    assert len(used) == len(set(used)) == sum((L + 127) // 128 for L in lens)
    assert n == len(used) + 4 and all(0 <= p < n for p in used)
    for b, L in enumerate(lens):  # a sequence's pages are the first entries of its row
        k = (L + 127) // 128
        assert (t[b, :k] >= 0).all() and (t[b, k:] == -1).all()
    with pytest.raises(ValueError):
        inputs.page_table([1000], 128, 7)


@pytest.mark.parametrize("tokens_per_row", [1, 64])
def test_pages_round_trip(tokens_per_row):
    lens, P = [300, 0, 700], 256
    t, n = inputs.page_table(lens, P, 3, seed=1)
    rows = 768 // tokens_per_row
    x = torch.randn((3, 2, rows, 5))
    pool = inputs.to_pages(x, t, n, P, tokens_per_row)
    assert pool.shape == (n, 2, P // tokens_per_row, 5)
    y = inputs.from_pages(pool, t, rows, tokens_per_row)
    for b, L in enumerate(lens):
        k = (L + P - 1) // P * P // tokens_per_row  # rows on the sequence's pages
        assert torch.equal(y[b, :, :k], x[b, :, :k]) and not y[b, :, k:].any()
    # the row of token t of sequence b sits at row t mod P of its page
    b, tok = 2, 517
    assert torch.equal(pool[t[b, tok // P], :, (tok % P) // tokens_per_row], x[b, :, tok // tokens_per_row])


def _paged(d, P=256, max_pages=16, num_pages=64, table=4096):
    d.page_table, d.page_tokens, d.max_pages, d.num_pages = table, P, max_pages, num_pages
    return d


@pytest.mark.parametrize("kw,want", [
    (dict(P=192), -1),                      # not whole 128-token slots
    (dict(P=384), -1),                      # not a power of two
    (dict(P=0), -1),
    (dict(max_pages=15), -1),               # the table row is short of max_seq_len = 4096
    (dict(max_pages=0), -1),
    (dict(num_pages=0), -1),
    (dict(table=4098), -2),                 # int32 table misaligned
])
def test_paged_descriptor_rules(lib, kw, want):
    null = ctypes.c_void_p(0)
    d = _paged(_desc(), **kw)
    assert lib.lbkv_decode_attn(ctypes.byref(d), *([null] * 8), 2, 0, 0, 128, null, null) == want
    assert lib.lbkv_workspace_bytes(ctypes.byref(d), 2, 0, 0, 128) == 0
    assert lib.lbkv_pack(ctypes.byref(d), null, null, 2, 0, 128, null, null, null, null) == want
    st = lib.lbkv_append(ctypes.byref(d), null, null, null, 2, 0, 0, 128, *([null] * 6), null)
    assert st == want


def test_valid_paged_descriptor_passes_the_format_checks(lib):
    null = ctypes.c_void_p(0)
    d = _paged(_desc(B=0))
    assert lib.lbkv_pack(ctypes.byref(d), null, null, 2, 1, 128, null, null, null, null) == 0
    assert lib.lbkv_append(ctypes.byref(d), null, null, null, 4, 0, 0, 64, *([null] * 6), null) == 0
    d = _paged(_desc())
    # past the paged checks: a GPU-less host stops at the device query, a GPU host at the NULL pointers
    assert lib.lbkv_decode_attn(ctypes.byref(d), *([null] * 8), 2, 0, 0, 128, null, null) not in (0, -3)


def test_bf16_comparator_has_no_paged_cache(lib):
    d = _paged(_desc())
    assert lib.lbkv_bf16_workspace_bytes(ctypes.byref(d)) == 0
    null = ctypes.c_void_p(0)
    assert lib.lbkv_decode_bf16(ctypes.byref(d), *([null] * 5), null) == -3


# ------------------------------------------------------------------ GPU

@pytest.fixture(scope="module")
def lbkv():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import bit_kv_cache_split_gb300 as m

    m.build.build()
    m.load()
    oracle.build()
    return m


def _rows(layout, g):
    return 1 if layout == oracle.TOKENWISE else g


def _page_cache(t, wl, table, num_pages, P):
    """The cache tensors of generated inputs t as page pools (on the GPU)."""
    out = {}
    for side, layout in (("k", wl.k_layout), ("v", wl.v_layout)):
        out[f"{side}_codes"] = inputs.to_pages(t[f"{side}_codes"].cuda(), table, num_pages, P)
        for part in ("scale", "off"):
            out[f"{side}_{part}"] = inputs.to_pages(t[f"{side}_{part}"].cuda(), table, num_pages, P,
                                                    _rows(layout, wl.group))
    return out


def _decode(m, t, wl, cache, ws, **kw):
    win = {}
    if "k_win" in t:
        win = dict(k_win=t["k_win"].cuda(), v_win=t["v_win"].cuda(), win_lens=t["win_lens"].cuda())
    out = m.decode_attn(t["q"].cuda(), cache["k_codes"], cache["k_scale"], cache["k_off"], cache["v_codes"],
                        cache["v_scale"], cache["v_off"], t["seq_lens"].cuda(), bits=wl.bits, k_layout=wl.k_layout,
                        v_layout=wl.v_layout, group=wl.group, workspace=ws, **win, **kw)
    torch.cuda.synchronize()
    return out


def _workspace(m, wl):
    n = m.workspace_bytes(wl.batch, wl.num_q_heads, wl.num_kv_heads, wl.t_cap, wl.bits, wl.k_layout, wl.v_layout,
                          wl.group, window=wl.window > 0)
    return m.alloc_workspace(n, "cuda")


def _check_paged_decode(m, wl, P):
    t = inputs.generate(wl, "cpu")
    max_pages = wl.t_cap // P + (1 if wl.t_cap % P else 0)
    table, num_pages = inputs.page_table(wl.lens, P, max_pages, seed=wl.seed + 7)
    ws = _workspace(m, wl)
    contiguous = {k: t[k].cuda() for k in ("k_codes", "k_scale", "k_off", "v_codes", "v_scale", "v_off")}
    ref = _decode(m, t, wl, contiguous, ws)
    got = _decode(m, t, wl, _page_cache(t, wl, table, num_pages, P), ws, page_table=table.cuda(),
                  max_seq_len=wl.t_cap)
    assert m.device_status(ws) == 0
    assert torch.equal(got.view(torch.int16), ref.view(torch.int16)), wl.name
    return got, t


@pytest.mark.gpu
@pytest.mark.parametrize("bits", [2, 4])
@pytest.mark.parametrize("kl,vl", [(0, 0), (1, 0), (0, 1), (1, 1)])
@pytest.mark.parametrize("P", [128, 256])
def test_paged_decode_equals_contiguous(lbkv, bits, kl, vl, P):
    s = (0.01, 0.1) if bits == 2 else (0.002, 0.02)
    wl = inputs.Workload(f"paged-b{bits}-k{kl}-v{vl}-P{P}", 3, 8, 2, [300, 1000, 129], bits=bits, k_layout=kl,
                         v_layout=vl, group=128, s_range=s, seed=11)
    got, t = _check_paged_decode(lbkv, wl, P)
    ref = oracle.decode_ref(oracle.inputs_from_tensors(t, bits=bits, k_layout=kl, v_layout=vl, group=128, Hkv=2,
                                                       T_cap=wl.t_cap))
    from tests.test_decode_gpu import assert_parity

    assert_parity(got.float().cpu().numpy().astype(np.float64), ref, wl.name)


@pytest.mark.gpu
@pytest.mark.parametrize("bits,kl,vl,g,hq", [(2, 0, 0, 32, 8), (2, 1, 0, 64, 4), (4, 0, 1, 32, 2), (2, 0, 0, 64, 1),
                                             (4, 1, 1, 64, 8), (2, 0, 1, 32, 4)])
def test_paged_decode_groups_and_gqa(lbkv, bits, kl, vl, g, hq):
    s = (0.01, 0.1) if bits == 2 else (0.002, 0.02)
    wl = inputs.Workload(f"paged-g{g}-hq{hq}", 4, 2 * hq, 2, [1, 640, 255, 0], bits=bits, k_layout=kl, v_layout=vl,
                         group=g, s_range=s, seed=12)
    _check_paged_decode(lbkv, wl, 128)


@pytest.mark.gpu
def test_paged_decode_with_window_and_long_pages(lbkv):
    wl = inputs.Workload("paged-window", 2, 16, 4, [3000, 77], bits=2, k_layout=1, v_layout=0, group=128,
                         s_range=(0.01, 0.1), window=40, seed=13)
    _check_paged_decode(lbkv, wl, 512)


@pytest.mark.gpu
def test_paged_decode_full_size_headline_shape(lbkv):
    """Batch 32 at 32K tokens, 32q/8kv, INT2 token-wise g128 over 128-token pages."""
    _check_paged_decode(lbkv, inputs.decode_int2(32, 32768), 128)


@pytest.mark.gpu
def test_bad_page_entry_is_reported_and_read_as_page_zero(lbkv):
    wl = inputs.Workload("paged-bad", 2, 8, 2, [300, 200], bits=2, group=128, s_range=(0.01, 0.1), seed=14)
    t = inputs.generate(wl, "cpu")
    table, num_pages = inputs.page_table(wl.lens, 128, 3, seed=3)
    cache = _page_cache(t, wl, table, num_pages, 128)
    ws = _workspace(lbkv, wl)
    bad = table.clone()
    bad[0, 1] = num_pages  # outside the pool
    out = _decode(lbkv, t, wl, cache, ws, page_table=bad.cuda(), max_seq_len=384)
    assert lbkv.device_status(ws) == 5
    assert torch.isfinite(out.float()).all()
    # the same call with page 0 in that entry gives the same output
    zero = table.clone()
    zero[0, 1] = 0
    again = _decode(lbkv, t, wl, cache, ws, page_table=zero.cuda(), max_seq_len=384)
    assert lbkv.device_status(ws) == 0
    assert torch.equal(out.view(torch.int16), again.view(torch.int16))


@pytest.mark.gpu
@pytest.mark.parametrize("bits", [2, 4])
@pytest.mark.parametrize("layout", [0, 1])
@pytest.mark.parametrize("g,P", [(128, 128), (32, 256), (64, 128)])
def test_paged_pack_stores_the_contiguous_rows(lbkv, bits, layout, g, P):
    lens = [0, 130, 1000, 256]
    x, sl = inputs.generate_pack_source(4, 2, lens, seed=21)
    x, sl = x.cuda(), sl.cuda()
    T = x.shape[2]
    table, num_pages = inputs.page_table(lens, P, (T + P - 1) // P, seed=22)
    ws = lbkv.alloc_workspace(256, "cuda")
    pc, ps, pz = lbkv.pack(x, sl, bits=bits, layout=layout, group=g, page_table=table.cuda(), num_pages=num_pages,
                           page_tokens=P, workspace=ws)
    assert lbkv.device_status(ws) == 0
    r = _rows(layout, g)
    got = [inputs.from_pages(a, table, T // rr) for a, rr in ((pc, 1), (ps, r), (pz, r))]
    rc, rs, rz = oracle.pack(bits16(x), np.asarray(lens, np.int32), bits, layout, g)
    for b, L in enumerate(lens):
        n = L if layout == 0 else (L + g - 1) // g
        assert np.array_equal(got[0][b, :, :L].cpu().numpy(), rc[b, :, :L]), ("codes", b)
        assert np.array_equal(bits16(got[1][b, :, :n]), rs[b, :, :n]), ("scale", b)
        assert np.array_equal(bits16(got[2][b, :, :n]), rz[b, :, :n]), ("offset", b)
    # the spare pages (named by no entry) are not touched
    used = set(table[table >= 0].tolist())
    spare = [p for p in range(num_pages) if p not in used]
    assert not pc[spare].any() and not ps[spare].any()


@pytest.mark.gpu
def test_paged_pack_bad_page_entry(lbkv):
    lens = [200]
    x, sl = inputs.generate_pack_source(1, 2, lens, seed=23)
    table = torch.tensor([[1, 9]], dtype=torch.int32)  # pool of 2 pages: the second entry is outside
    ws = lbkv.alloc_workspace(256, "cuda")
    pc, _, _ = lbkv.pack(x.cuda(), sl.cuda(), bits=2, layout=0, group=128, page_table=table.cuda(), num_pages=2,
                         page_tokens=128, workspace=ws)
    assert lbkv.device_status(ws) == 5
    assert pc[1].any() and not pc[0].any()  # the first page is stored, nothing is written for the bad one


def _token(x, pos):
    T = x.shape[2]
    return torch.stack([x[b, :, min(p, T - 1)] for b, p in enumerate(pos)]).contiguous()


@pytest.mark.gpu
@pytest.mark.parametrize("bits", [2, 4])
@pytest.mark.parametrize("kl,vl,g", [(0, 0, 128), (0, 0, 32), (1, 0, 64), (1, 1, 128), (0, 1, 32)])
def test_paged_append_equals_packing_the_history(lbkv, bits, kl, vl, g):
    B, Hkv, T, P = 3, 2, 512, 256
    lens0 = [0, g, 2 * g]
    n = g + 3
    gen = torch.Generator().manual_seed(31)
    xk = torch.randn((B, Hkv, T, D), generator=gen).to(torch.bfloat16).cuda()
    xv = torch.randn((B, Hkv, T, D), generator=gen).to(torch.bfloat16).cuda()
    table, num_pages = inputs.page_table([T] * B, P, T // P, seed=32)
    tab = table.cuda()
    l0 = torch.tensor(lens0, dtype=torch.int32, device="cuda")
    kw = dict(page_table=tab, num_pages=num_pages, page_tokens=P)
    k = lbkv.pack(xk, l0, bits=bits, layout=kl, group=g, **kw)
    v = lbkv.pack(xv, l0, bits=bits, layout=vl, group=g, **kw)
    windowed = kl == 1 or vl == 1
    win = {}
    if windowed:
        win = dict(k_win=torch.zeros((B, Hkv, 128, D), dtype=torch.bfloat16, device="cuda"),
                   v_win=torch.zeros((B, Hkv, 128, D), dtype=torch.bfloat16, device="cuda"),
                   win_lens=torch.zeros((B,), dtype=torch.int32, device="cuda"))
    lens = l0.clone()
    ws = lbkv.alloc_workspace(256, "cuda")
    pos = list(lens0)
    for _ in range(n):
        lbkv.append(_token(xk, pos), _token(xv, pos), lens, *k, *v, bits=bits, k_layout=kl, v_layout=vl, group=g,
                    page_table=tab, max_seq_len=T, workspace=ws, **win)
        pos = [p + 1 for p in pos]
    torch.cuda.synchronize()
    assert lbkv.device_status(ws) == 0
    final = [L + (g if windowed else n) for L in lens0]
    assert lens.cpu().tolist() == final
    for (c, s, z), x, layout in ((k, xk, kl), (v, xv, vl)):
        r = _rows(layout, g)
        cc, ss, zz = (inputs.from_pages(a, table, T // rr) for a, rr in ((c, 1), (s, r), (z, r)))
        rc, rs, rz = oracle.pack(bits16(x), np.asarray(final, np.int32), bits, layout, g)
        for b, L in enumerate(final):
            m = L if layout == 0 else (L + g - 1) // g
            assert np.array_equal(cc[b, :, :L].cpu().numpy(), rc[b, :, :L]), ("codes", b)
            assert np.array_equal(bits16(ss[b, :, :m]), rs[b, :, :m]), ("scale", b)
            assert np.array_equal(bits16(zz[b, :, :m]), rz[b, :, :m]), ("offset", b)
    # and the grown paged cache decodes like its contiguous gather
    q = torch.randn((B, 4 * Hkv, D), generator=gen).to(torch.bfloat16).cuda()
    common = dict(bits=bits, k_layout=kl, v_layout=vl, group=g, **win)
    got = lbkv.decode_attn(q, *k, *v, lens, page_table=tab, max_seq_len=T, **common)
    kc = [inputs.from_pages(a, table, T // rr) for a, rr in ((k[0], 1), (k[1], _rows(kl, g)), (k[2], _rows(kl, g)))]
    vc = [inputs.from_pages(a, table, T // rr) for a, rr in ((v[0], 1), (v[1], _rows(vl, g)), (v[2], _rows(vl, g)))]
    ref = lbkv.decode_attn(q, *kc, *vc, lens, **common)
    torch.cuda.synchronize()
    assert torch.equal(got.view(torch.int16), ref.view(torch.int16))


@pytest.mark.gpu
def test_paged_append_bad_page_entry_changes_nothing(lbkv):
    B, Hkv, P = 2, 2, 128
    table = torch.tensor([[0, 1], [2, 7]], dtype=torch.int32)  # pool of 3 pages; entry [1][1] is outside
    pool = [torch.zeros((3, Hkv, P, 32), dtype=torch.uint8, device="cuda")]
    pool += [torch.zeros((3, Hkv, P, 1), dtype=torch.float16, device="cuda") for _ in range(2)]
    vpool = [t.clone() for t in pool]
    lens = torch.tensor([5, 128], dtype=torch.int32, device="cuda")  # sequence 1 appends into page entry 1
    x = torch.randn((B, Hkv, D)).to(torch.bfloat16).cuda()
    ws = lbkv.alloc_workspace(256, "cuda")
    lbkv.append(x, x, lens, *pool, *vpool, bits=2, group=128, page_table=table.cuda(), workspace=ws)
    assert lbkv.device_status(ws) == 5
    assert lens.cpu().tolist() == [6, 128]
    assert pool[0][0, :, 5].any() and not pool[0][1:].any()
