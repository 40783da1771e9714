"""The CUDA quantizer (lbkv_pack) is bit-exact with the oracle's, and a packed
cache decodes to the oracle's output on that same packed cache."""

import numpy as np
import pytest
import torch

import oracle
from bit_kv_cache_split_gb300 import inputs
from tests.helpers import bits16, to_oracle
from tests.test_decode_gpu import assert_parity, lbkv  # noqa: F401  (fixture)

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("bits", [2, 4])
@pytest.mark.parametrize("layout", [0, 1])
@pytest.mark.parametrize("g", [32, 64, 128])
def test_pack_bit_exact(lbkv, bits, layout, g):
    x, lens = inputs.generate_pack_source(3, 2, [515, 128, 1], seed=2)
    x = x * 3.0
    x = x.to(torch.bfloat16)
    sentinel = 0x1234
    B, H, T, D = x.shape
    sshape = (B, H, T, D // g) if layout == 0 else (B, H, T // g, D)
    s0 = torch.full(sshape, sentinel, dtype=torch.int16).view(torch.float16)
    codes, s, z = lbkv.pack(x.cuda(), lens.cuda(), bits=bits, layout=layout, group=g, scale=s0.clone().cuda(),
                            off=s0.clone().cuda())
    torch.cuda.synchronize()
    rc, rs, rz = oracle.pack(bits16(x), lens.numpy(), bits, layout, g,
                             scale_init=np.full(sshape, sentinel, np.uint16), off_init=np.full(sshape, sentinel, np.uint16))
    assert np.array_equal(codes.cpu().numpy(), rc)
    assert np.array_equal(bits16(s), rs)
    assert np.array_equal(bits16(z), rz)


def test_pack_special_values(lbkv):
    """Constant groups, exact ties, signed zeros and large magnitudes."""
    rng = np.random.default_rng(5)
    T, D = 128, 128
    x = rng.standard_normal((1, 1, T, D)).astype(np.float32)
    x[0, 0, 0] = 0.75                       # constant token
    x[0, 0, 1, :4] = [0, 0.5, 1.5, 3]       # ties inside a group
    x[0, 0, 2] = 0.0
    x[0, 0, 2, ::2] = -0.0                  # signed zeros
    x[0, 0, 3] *= 1000.0
    xt = torch.from_numpy(x).to(torch.bfloat16)
    lens = torch.tensor([T], dtype=torch.int32)
    for bits in (2, 4):
        for layout, g in ((0, 32), (0, 128), (1, 128)):
            codes, s, z = lbkv.pack(xt.cuda(), lens.cuda(), bits=bits, layout=layout, group=g)
            rc, rs, rz = oracle.pack(bits16(xt), lens.numpy(), bits, layout, g)
            assert np.array_equal(codes.cpu().numpy(), rc), (bits, layout, g)
            assert np.array_equal(bits16(s), rs) and np.array_equal(bits16(z), rz), (bits, layout, g)


@pytest.mark.parametrize("bits", [2, 4])
@pytest.mark.parametrize("kl,vl", [(0, 0), (1, 0), (0, 1), (1, 1)])
def test_quantize_then_decode(lbkv, bits, kl, vl):
    """bf16 K/V ~ N(0, 1) -> lbkv_pack -> lbkv_decode_attn, against the oracle on the packed cache."""
    B, Hkv, hq, g = 2, 2, 4, 128
    lens = [700, 259]
    k, lt = inputs.generate_pack_source(B, Hkv, lens, seed=2)
    v, _ = inputs.generate_pack_source(B, Hkv, lens, seed=12)
    q = torch.randn((B, Hkv * hq, 128), generator=torch.Generator().manual_seed(22)).to(torch.bfloat16)
    kc, ks, kz = lbkv.pack(k.cuda(), lt.cuda(), bits=bits, layout=kl, group=g)
    vc, vs, vz = lbkv.pack(v.cuda(), lt.cuda(), bits=bits, layout=vl, group=g)
    out = lbkv.decode_attn(q.cuda(), kc, ks, kz, vc, vs, vz, lt.cuda(), bits=bits, k_layout=kl, v_layout=vl, group=g)
    torch.cuda.synchronize()
    wl = inputs.Workload("packed", B, Hkv * hq, Hkv, lens, bits=bits, k_layout=kl, v_layout=vl, group=g)
    t = dict(q=q, k_codes=kc.cpu(), k_scale=ks.cpu(), k_off=kz.cpu(), v_codes=vc.cpu(), v_scale=vs.cpu(),
             v_off=vz.cpu(), seq_lens=lt)
    ref = oracle.decode_ref(to_oracle(t, wl))
    assert_parity(out.float().cpu().numpy().astype(np.float64), ref, f"packed b{bits} k{kl} v{vl}")


def test_quantize_then_decode_full_size_int4(lbkv):
    """bf16 K/V ~ N(0, 1) at the INT4 decode shape (batch 8, 8 KV heads, 32 query heads,
    32K context) -> lbkv_pack (token-wise, g128) -> lbkv_decode_attn, against the oracle on
    the packed cache of sampled (sequence, KV head) units."""
    B, Hkv, Hq, T, g = 8, 8, 32, 32768, 128
    hq = Hq // Hkv
    k, lens = inputs.generate_pack_source(B, Hkv, T, seed=2, device="cuda")
    v, _ = inputs.generate_pack_source(B, Hkv, T, seed=12, device="cuda")
    q = torch.randn((B, Hq, 128), generator=torch.Generator().manual_seed(22)).to(torch.bfloat16)
    kc, ks, kz = lbkv.pack(k, lens, bits=4, layout=0, group=g)
    vc, vs, vz = lbkv.pack(v, lens, bits=4, layout=0, group=g)
    del k, v
    out = lbkv.decode_attn(q.cuda(), kc, ks, kz, vc, vs, vz, lens, bits=4, group=g)
    torch.cuda.synchronize()
    got_all = out.float().cpu().numpy().astype(np.float64)
    for b, kvh in [(0, 0), (3, 5), (7, 7)]:
        sl = lambda x: x[b:b + 1, kvh:kvh + 1].contiguous().cpu()  # noqa: E731
        t = dict(q=q[b:b + 1, kvh * hq:(kvh + 1) * hq].contiguous(), k_codes=sl(kc), k_scale=sl(ks), k_off=sl(kz),
                 v_codes=sl(vc), v_scale=sl(vs), v_off=sl(vz), seq_lens=torch.tensor([T], dtype=torch.int32))
        wl = inputs.Workload("packed-int4-b8-ctx32768", 1, hq, 1, [T], bits=4, group=g)
        ref = oracle.decode_ref(to_oracle(t, wl))[0]
        assert_parity(got_all[b, kvh * hq:(kvh + 1) * hq], ref, f"packed INT4 full size unit ({b},{kvh})")


@pytest.mark.parametrize("bits", [2, 4])
@pytest.mark.parametrize("layout", [0, 1])
def test_pack_quotients_at_rounding_boundaries(lbkv, bits, layout):
    """Inputs whose quotients (x - z) / s fall exactly on, or within an ulp of, the
    half-integers where the rounding of a code changes: every group spans 0 .. 2^b - 1 (so
    s = 1 exactly) plus small bf16 perturbations, and the remaining channels sit on the
    half-integers (exact ties, rounded to even) and on their bf16 neighbours."""
    rng = np.random.default_rng(11 + bits + layout)
    qmax = (1 << bits) - 1
    T, D = 256, 128
    base = rng.integers(0, qmax, (1, 2, T, D)).astype(np.float32) + 0.5        # exact half-integers
    nudge = rng.choice([-1, 0, 0, 1], size=base.shape).astype(np.float32)
    x = (torch.from_numpy(base).to(torch.bfloat16).view(torch.int16) + torch.from_numpy(nudge).to(torch.int16))
    x = x.view(torch.bfloat16).float().numpy()
    if layout == 0:
        x[..., 0::32] = 0.0          # each group of 32 channels (and of 64, 128) spans [0, qmax]
        x[..., 1::32] = float(qmax)
    else:
        x[:, :, 0::32, :] = 0.0      # each token group spans [0, qmax] per channel
        x[:, :, 1::32, :] = float(qmax)
    x[0, 1] *= 0.37                  # a second head with an inexact scale
    xt = torch.from_numpy(x).to(torch.bfloat16)
    lens = torch.tensor([T], dtype=torch.int32)
    for g in (32, 128):
        codes, s, z = lbkv.pack(xt.cuda(), lens.cuda(), bits=bits, layout=layout, group=g)
        rc, rs, rz = oracle.pack(bits16(xt), lens.numpy(), bits, layout, g)
        assert np.array_equal(codes.cpu().numpy(), rc), (bits, layout, g)
        assert np.array_equal(bits16(s), rs) and np.array_equal(bits16(z), rz), (bits, layout, g)
