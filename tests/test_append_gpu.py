"""Quantize-on-append (lbkv_append) against the oracle.

A cache grown one token at a time equals the oracle's quantizer applied to the whole
bf16 history, bit for bit. Channel-wise sides gather their tokens in the bf16 window and
close a group when it holds `group` tokens. A token that does not fit changes nothing
and is reported. A grown cache (with its window) decodes to the oracle's output."""

import numpy as np
import pytest
import torch

import oracle
from bit_kv_cache_split_gb300 import inputs
from tests.helpers import bits16
from tests.test_decode_gpu import assert_parity, lbkv  # noqa: F401  (fixture)

pytestmark = pytest.mark.gpu

D = 128


def _history(B, Hkv, T, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn((B, Hkv, T, D), generator=g).to(torch.bfloat16)


def _token(x, pos):
    """x [B][Hkv][T][D] (device) at position pos[b] of each sequence -> [B][Hkv][D] (a full
    sequence gets its last token again: it is not stored)."""
    T = x.shape[2]
    return torch.stack([x[b, :, min(p, T - 1)] for b, p in enumerate(pos)]).contiguous()


def _check_side(codes, scale, off, x, lens, bits, layout, g):
    """Valid codes, scales and offsets equal the oracle's packing of the history."""
    rc, rs, rz = oracle.pack(bits16(x), np.asarray(lens, np.int32), bits, layout, g)
    c, s, z = codes.cpu().numpy(), bits16(scale), bits16(off)
    for b, L in enumerate(lens):
        assert np.array_equal(c[b, :, :L], rc[b, :, :L]), ("codes", b)
        n = L if layout == 0 else (L + g - 1) // g
        assert np.array_equal(s[b, :, :n], rs[b, :, :n]), ("scale", b)
        assert np.array_equal(z[b, :, :n], rz[b, :, :n]), ("offset", b)


class Cache:
    """A packed cache of the first lens0 tokens of bf16 histories xk, xv, on the GPU."""

    def __init__(self, lbkv, xk, xv, lens0, bits, kl, vl, g, window=False):
        self.bits, self.kl, self.vl, self.g = bits, kl, vl, g
        self.xk, self.xv = xk.cuda(), xv.cuda()
        l0 = torch.tensor(lens0, dtype=torch.int32).cuda()
        self.k = lbkv.pack(self.xk, l0, bits=bits, layout=kl, group=g)
        self.v = lbkv.pack(self.xv, l0, bits=bits, layout=vl, group=g)
        self.lens = l0.clone()
        B, Hkv = xk.shape[:2]
        self.win = None
        if window:
            self.win = (torch.zeros((B, Hkv, 128, D), dtype=torch.bfloat16, device="cuda"),
                        torch.zeros((B, Hkv, 128, D), dtype=torch.bfloat16, device="cuda"),
                        torch.zeros((B,), dtype=torch.int32, device="cuda"))
        self.next = list(lens0)  # history position of each sequence's next token

    def append(self, lbkv, n, workspace=None):
        for _ in range(n):
            kw = {}
            if self.win is not None:
                kw = dict(k_win=self.win[0], v_win=self.win[1], win_lens=self.win[2])
            lbkv.append(_token(self.xk, self.next), _token(self.xv, self.next), self.lens, *self.k, *self.v,
                        bits=self.bits, k_layout=self.kl, v_layout=self.vl, group=self.g, workspace=workspace, **kw)
            self.next = [p + 1 for p in self.next]
        torch.cuda.synchronize()


@pytest.mark.parametrize("bits", [2, 4])
@pytest.mark.parametrize("g", [32, 64, 128])
def test_append_tokenwise_equals_packing_the_history(lbkv, bits, g):
    lens0, n = [0, 5, 100], 21
    xk, xv = _history(3, 2, 256, 40), _history(3, 2, 256, 41)
    c = Cache(lbkv, xk, xv, lens0, bits, 0, 0, g)
    c.append(lbkv, n)
    final = [L + n for L in lens0]
    assert c.lens.cpu().tolist() == final
    _check_side(*c.k, xk, final, bits, 0, g)
    _check_side(*c.v, xv, final, bits, 0, g)


@pytest.mark.parametrize("bits", [2, 4])
@pytest.mark.parametrize("g", [32, 64, 128])
@pytest.mark.parametrize("kl,vl", [(1, 0), (0, 1), (1, 1)])
def test_append_channelwise_closes_groups_through_the_window(lbkv, bits, g, kl, vl):
    lens0, rest = [0, g], 5
    xk, xv = _history(2, 2, 512, 42), _history(2, 2, 512, 43)
    c = Cache(lbkv, xk, xv, lens0, bits, kl, vl, g, window=True)
    c.append(lbkv, g + rest)
    final = [L + g for L in lens0]
    assert c.lens.cpu().tolist() == final
    assert c.win[2].cpu().tolist() == [rest] * 2
    _check_side(*c.k, xk, final, bits, kl, g)
    _check_side(*c.v, xv, final, bits, vl, g)
    # the window holds the last `rest` tokens, exact bf16 copies
    for side, x in ((0, xk), (1, xv)):
        w = c.win[side].cpu()
        for b, L in enumerate(final):
            assert torch.equal(w[b, :, :rest].view(torch.int16), x[b, :, L:L + rest].view(torch.int16))


def test_append_that_does_not_fit_changes_nothing(lbkv):
    g, T = 128, 256
    xk, xv = _history(2, 2, T, 44), _history(2, 2, T, 45)
    c = Cache(lbkv, xk, xv, [T, 3], 2, 0, 0, g)
    k_before = [t.clone() for t in c.k]
    ws = torch.zeros(64, dtype=torch.int32, device="cuda")
    c.append(lbkv, 1, workspace=ws)
    assert c.lens.cpu().tolist() == [T, 4]  # the full sequence is left as it was
    assert torch.equal(c.k[0][0], k_before[0][0]) and torch.equal(c.k[1][0], k_before[1][0])
    assert lbkv.device_status(ws) == 4
    assert lbkv.device_status(ws) == 0  # read and cleared


def test_append_channelwise_needs_whole_groups(lbkv):
    """A channel-wise cache whose length is not a multiple of the group cannot close the next group."""
    g = 64
    xk, xv = _history(1, 2, 256, 46), _history(1, 2, 256, 47)
    c = Cache(lbkv, xk, xv, [10], 2, 1, 0, g, window=True)
    ws = torch.zeros(64, dtype=torch.int32, device="cuda")
    c.append(lbkv, g - 1, workspace=ws)  # fills the window up to one short of a group
    assert c.win[2].cpu().tolist() == [g - 1] and lbkv.device_status(ws) == 0
    c.append(lbkv, 1, workspace=ws)  # the group cannot be closed at position 10
    assert c.lens.cpu().tolist() == [10] and c.win[2].cpu().tolist() == [g - 1]
    assert lbkv.device_status(ws) == 4


@pytest.mark.parametrize("bits", [2, 4])
@pytest.mark.parametrize("kl,vl", [(0, 0), (1, 0), (0, 1), (1, 1)])
def test_decode_after_appends_matches_oracle(lbkv, bits, kl, vl):
    B, Hkv, hq, g, T = 2, 2, 4, 128, 512
    lens0 = [128, 256]
    n = g + 5
    xk, xv = _history(B, Hkv, T, 48), _history(B, Hkv, T, 49)
    windowed = kl == 1 or vl == 1
    c = Cache(lbkv, xk, xv, lens0, bits, kl, vl, g, window=windowed)
    c.append(lbkv, n)
    q = (torch.randn((B, Hkv * hq, D), generator=torch.Generator().manual_seed(50))).to(torch.bfloat16)
    kw = dict(k_win=c.win[0], v_win=c.win[1], win_lens=c.win[2]) if windowed else {}
    out = lbkv.decode_attn(q.cuda(), *c.k, *c.v, c.lens, bits=bits, k_layout=kl, v_layout=vl, group=g, **kw)
    torch.cuda.synchronize()
    t = dict(q=q, k_codes=c.k[0].cpu(), k_scale=c.k[1].cpu(), k_off=c.k[2].cpu(), v_codes=c.v[0].cpu(),
             v_scale=c.v[1].cpu(), v_off=c.v[2].cpu(), seq_lens=c.lens.cpu())
    if windowed:
        t.update(k_win=c.win[0].cpu(), v_win=c.win[1].cpu(), win_lens=c.win[2].cpu())
    ref = oracle.decode_ref(oracle.inputs_from_tensors(t, bits=bits, k_layout=kl, v_layout=vl, group=g, Hkv=Hkv,
                                                       T_cap=T))
    assert_parity(out.float().cpu().numpy().astype(np.float64), ref, f"appended b{bits} k{kl} v{vl}")
    expect = [L + (g if windowed else n) for L in lens0]
    assert c.lens.cpu().tolist() == expect
