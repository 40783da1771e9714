"""Parity of the tensor-core decode kernel (QK^T on tcgen05, selected with
LBKV_DECODE_KERNEL=tc for a token-wise K side) with the fp64 oracle.

Same bar as the default kernel: bf16 output within max-abs 5e-3 and relative L2
3e-3 of the oracle run on the same quantized cache, over INT2 and INT4, token-wise
and channel-wise V sides, GQA 1..8, groups 32/64/128, ragged lengths ending
mid-item, empty sequences, a bf16 window, a paged and a rotated cache, and the
benchmark's full-size headline shape on sampled (sequence, KV head) units."""

import numpy as np
import pytest
import torch

import oracle
from bit_kv_cache_split_gb300 import inputs
from tests.helpers import to_oracle
from tests.test_decode_gpu import _wl, assert_parity, check, lbkv, run_gpu, sampled_parity  # noqa: F401

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def tc_kernel(monkeypatch):
    monkeypatch.setenv("LBKV_DECODE_KERNEL", "tc")


def test_tc_tiny(lbkv):
    check(lbkv, inputs.tiny_int2())


@pytest.mark.parametrize("bits", [2, 4])
@pytest.mark.parametrize("vl", [0, 1])
def test_tc_layouts(lbkv, bits, vl):
    check(lbkv, _wl(bits, 0, vl, seed=70 + 10 * bits + vl))


@pytest.mark.parametrize("bits", [2, 4])
@pytest.mark.parametrize("hq", [1, 2, 4, 8])
def test_tc_gqa(lbkv, bits, hq):
    check(lbkv, _wl(bits, 0, 0, hq=hq, lens=(777, 64), seed=80 + hq))


@pytest.mark.parametrize("g,hq,vl", [(64, 1, 0), (64, 4, 0), (64, 8, 0), (32, 1, 0), (32, 2, 0), (32, 4, 0),
                                     (64, 4, 1), (64, 8, 1), (32, 2, 1)])
def test_tc_groups(lbkv, g, hq, vl):
    check(lbkv, _wl(2, 0, vl, g=g, hq=hq, lens=(513, 95), seed=90 + g + hq + vl))


def test_tc_window_and_empty(lbkv):
    wl = _wl(2, 0, 0, lens=(600, 0, 37), seed=95, window=128)
    t = inputs.generate(wl, "cpu")
    t["win_lens"] = torch.tensor([128, 17, 0], dtype=torch.int32)
    got = run_gpu(lbkv, t, wl)
    assert_parity(got, oracle.decode_ref(to_oracle(t, wl)), "tc window")


def test_tc_peaked_softmax(lbkv):
    """Large scores: the running maximum is raised lazily (by more than 2^8 only)."""
    check(lbkv, _wl(2, 0, 0, lens=(2000, 333), seed=96, q_std=6.0, sm_scale=0.5))


def test_tc_rotated(lbkv):
    wl = _wl(2, 0, 0, lens=(900, 130), seed=97)
    t = inputs.generate(wl, "cpu")
    got = run_gpu(lbkv, t, wl, rotation=3)
    x = to_oracle(t, wl)
    x.rotation = 3
    assert_parity(got, oracle.decode_ref(x), "tc rotated")


def test_tc_paged_equals_contiguous(lbkv):
    wl = _wl(2, 0, 0, lens=(700, 129, 0), seed=98)
    t = {k: v.cuda() for k, v in inputs.generate(wl, "cpu").items()}
    P = 128
    table, n_pages = inputs.page_table(wl.lens, P, wl.t_cap // P, seed=99)
    pool = {k: inputs.to_pages(t[k], table, n_pages, P) for k in ("k_codes", "k_scale", "k_off", "v_codes", "v_scale",
                                                                  "v_off")}
    a = lbkv.decode_attn(t["q"], t["k_codes"], t["k_scale"], t["k_off"], t["v_codes"], t["v_scale"], t["v_off"],
                         t["seq_lens"], bits=2, group=128)
    b = lbkv.decode_attn(t["q"], pool["k_codes"], pool["k_scale"], pool["k_off"], pool["v_codes"], pool["v_scale"],
                         pool["v_off"], t["seq_lens"], bits=2, group=128, page_table=table.cuda(),
                         max_seq_len=wl.t_cap)
    torch.cuda.synchronize()
    assert torch.equal(a, b)


@pytest.mark.parametrize("batch,ctx", [(32, 32768), (1, 131072)])
def test_tc_full_size_sampled(lbkv, batch, ctx):
    wl = inputs.decode_int2(batch, ctx)
    sampled_parity(lbkv, wl, [(0, 0), (batch - 1, 7), (batch // 2, 3)])


def test_tc_no_device_status(lbkv):
    wl = _wl(4, 0, 1, lens=(1500, 3), seed=100)
    t = {k: v.cuda() for k, v in inputs.generate(wl, "cpu").items()}
    n = lbkv.workspace_bytes(wl.batch, wl.num_q_heads, wl.num_kv_heads, wl.t_cap, 4, 0, 1, 128)
    ws = lbkv._binding.alloc_workspace(n, "cuda")
    lbkv.decode_attn(t["q"], t["k_codes"], t["k_scale"], t["k_off"], t["v_codes"], t["v_scale"], t["v_off"],
                     t["seq_lens"], bits=4, v_layout=1, workspace=ws)
    assert lbkv.device_status(ws) == 0
