"""Parity of the CUDA decode path (through the C ABI) with the fp64 oracle.

Bar: bf16 output within max-abs 5e-3 and relative L2 3e-3 of the oracle run
on the same quantized cache, for every K/V layout pair at INT2 and INT4, over
ragged lengths that span several 128-token slots and end mid-slot, GQA 1..8,
groups 32/64/128, a bf16 window, empty sequences and peaked softmaxes; at
the full benchmark sizes on sampled (sequence, KV head) units."""

import time

import numpy as np
import pytest
import torch

import oracle
from bit_kv_cache_split_gb300 import inputs
from tests.helpers import to_oracle

pytestmark = pytest.mark.gpu

MAX_ABS = 5e-3
REL_L2 = 3e-3


@pytest.fixture(scope="module")
def lbkv():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import bit_kv_cache_split_gb300 as m

    m.build.build()
    m.load()
    oracle.build()
    return m


def run_gpu(m, t, wl, **kw):
    dev = {k: v.cuda() for k, v in t.items()}
    win = {}
    if "k_win" in dev:
        win = dict(k_win=dev["k_win"], v_win=dev["v_win"], win_lens=dev["win_lens"])
    out = m.decode_attn(dev["q"], dev["k_codes"], dev["k_scale"], dev["k_off"], dev["v_codes"], dev["v_scale"],
                        dev["v_off"], dev["seq_lens"], bits=wl.bits, k_layout=wl.k_layout, v_layout=wl.v_layout,
                        group=wl.group, sm_scale=wl.sm_scale, **win, **kw)
    torch.cuda.synchronize()
    return out.float().cpu().numpy().astype(np.float64)


def errors(got, ref):
    d = got - ref
    return float(np.max(np.abs(d))), float(np.linalg.norm(d) / max(np.linalg.norm(ref), 1e-30))


def assert_parity(got, ref, what=""):
    mx, rl2 = errors(got, ref)
    assert np.all(np.isfinite(got)), what
    assert mx <= MAX_ABS and rl2 <= REL_L2, f"{what}: max-abs {mx:.3e}, rel-L2 {rl2:.3e}"
    return mx, rl2


def check(m, wl, **kw):
    t = inputs.generate(wl, "cpu")
    got = run_gpu(m, t, wl, **kw)
    ref = oracle.decode_ref(to_oracle(t, wl))
    return assert_parity(got, ref, wl.name)


def _wl(bits, kl, vl, g=128, hq=4, lens=(300, 1000, 129), seed=0, **kw):
    s = (0.01, 0.1) if bits == 2 else (0.002, 0.02)
    return inputs.Workload(f"b{bits}-k{kl}-v{vl}-g{g}-hq{hq}", len(lens), 2 * hq, 2, list(lens), bits=bits,
                           k_layout=kl, v_layout=vl, group=g, s_range=s, seed=seed, **kw)


def test_tiny_int2_full_output(lbkv):
    """Batch 1, 1 KV head, 4 query heads, 512 tokens, INT2 token-wise g=128 (seed 0)."""
    check(lbkv, inputs.tiny_int2())


@pytest.mark.parametrize("bits", [2, 4])
@pytest.mark.parametrize("kl,vl", [(0, 0), (1, 0), (0, 1), (1, 1)])
def test_layout_pairs(lbkv, bits, kl, vl):
    check(lbkv, _wl(bits, kl, vl, seed=10 * bits + 2 * kl + vl))


@pytest.mark.parametrize("bits", [2, 4])
@pytest.mark.parametrize("hq", [1, 2, 4, 8])
def test_gqa_ratios(lbkv, bits, hq):
    check(lbkv, _wl(bits, 0, 0, hq=hq, lens=(777, 64), seed=hq))


@pytest.mark.parametrize("bits", [2, 4])
@pytest.mark.parametrize("g", [32, 64])
@pytest.mark.parametrize("kl,vl", [(0, 1), (1, 1), (1, 0), (0, 0)])
def test_group_sizes(lbkv, bits, g, kl, vl):
    check(lbkv, _wl(bits, kl, vl, g=g, lens=(513, 95), seed=g + bits))


@pytest.mark.parametrize("g,hq", [(64, 1), (64, 2), (64, 4), (64, 8), (32, 1), (32, 2), (32, 4)])
@pytest.mark.parametrize("kl", [0, 1])
def test_tokenwise_v_channel_groups_all_gqa(lbkv, g, hq, kl):
    """Token-wise V with 2 or 4 value channel groups: (query, group) output columns."""
    check(lbkv, _wl(2, kl, 0, g=g, hq=hq, lens=(400, 37), seed=7 + hq))


def test_window(lbkv):
    wl = _wl(2, 0, 0, lens=(600, 0, 37), seed=5, window=128)
    t = inputs.generate(wl, "cpu")
    t["win_lens"] = torch.tensor([128, 17, 0], dtype=torch.int32)
    got = run_gpu(lbkv, t, wl)
    ref = oracle.decode_ref(to_oracle(t, wl))
    assert_parity(got, ref, "window")


def test_empty_and_single_token_sequences(lbkv):
    wl = _wl(2, 0, 0, lens=(0, 1, 128, 129), seed=3)
    t = inputs.generate(wl, "cpu")
    got = run_gpu(lbkv, t, wl)
    assert np.all(got[0] == 0)
    assert_parity(got, oracle.decode_ref(to_oracle(t, wl)), "empty/single")


@pytest.mark.parametrize("kl,vl", [(0, 0), (1, 1)])
def test_peaked_softmax(lbkv, kl, vl):
    """Large scores: most weight on a few tokens, exercising the running maximum."""
    check(lbkv, _wl(2, kl, vl, lens=(2000, 333), seed=21, q_std=6.0, sm_scale=0.5))


def test_full_capacity_and_padding_garbage(lbkv):
    """seq_len == T_cap, and NaN patterns in padding scales must not leak."""
    wl = _wl(4, 0, 0, lens=(256, 130), seed=8)
    t = inputs.generate(wl, "cpu")
    t["k_scale"][1, :, 130:] = float("nan")
    t["v_scale"][1, :, 130:] = float("nan")
    t["v_off"][1, :, 130:] = float("inf")
    got = run_gpu(lbkv, t, wl)
    assert_parity(got, oracle.decode_ref(to_oracle(t, wl)), "padding")


def test_repeat_calls_are_bitwise_identical(lbkv):
    wl = _wl(2, 0, 0, lens=(3000, 17), seed=30)
    t = inputs.generate(wl, "cpu")
    a = run_gpu(lbkv, t, wl)
    b = run_gpu(lbkv, t, wl)
    assert np.array_equal(a, b)


def test_unsupported_combination_raises(lbkv):
    """Groups of 16 channels are not built."""
    wl = _wl(2, 0, 0, g=128, hq=4, lens=(10,))
    t = {k: v.cuda() for k, v in inputs.generate(wl, "cpu").items()}
    with pytest.raises(lbkv.LbkvError) as e:
        lbkv.decode_attn(t["q"], t["k_codes"], t["k_scale"], t["k_off"], t["v_codes"], t["v_scale"], t["v_off"],
                         t["seq_lens"], bits=2, group=16)
    assert e.value.status == -3


@pytest.mark.parametrize("bits", [2, 4])
@pytest.mark.parametrize("kl", [0, 1])
def test_tokenwise_v_four_groups_eight_queries(lbkv, bits, kl):
    """32 (query, V group) pairs per KV head: the queries of a KV head are split in two halves."""
    check(lbkv, _wl(bits, kl, 0, g=32, hq=8, lens=(700, 129, 0), seed=41 + bits + kl))


def test_tokenwise_v_four_groups_eight_queries_window(lbkv):
    wl = _wl(2, 0, 0, g=32, hq=8, lens=(300, 0), seed=43, window=64)
    t = inputs.generate(wl, "cpu")
    t["win_lens"] = torch.tensor([64, 5], dtype=torch.int32)
    got = run_gpu(lbkv, t, wl)
    assert_parity(got, oracle.decode_ref(to_oracle(t, wl)), "32 pairs + window")


def test_no_device_status_after_calls(lbkv):
    wl = _wl(2, 1, 0, lens=(900,), seed=31)
    t = {k: v.cuda() for k, v in inputs.generate(wl, "cpu").items()}
    n = lbkv.workspace_bytes(wl.batch, wl.num_q_heads, wl.num_kv_heads, wl.t_cap, 2, 1, 0, 128)
    ws = lbkv._binding.alloc_workspace(n, "cuda")
    lbkv.decode_attn(t["q"], t["k_codes"], t["k_scale"], t["k_off"], t["v_codes"], t["v_scale"], t["v_off"],
                     t["seq_lens"], bits=2, k_layout=1, workspace=ws)
    assert lbkv.device_status(ws) == 0


# ------------------------------------------------------------ full sizes

def unit_slice(t, wl, b, kvh):
    """The tensors of one (sequence, KV head) unit as a batch-1, 1-KV-head problem."""
    hq = wl.hq_per_kv
    sub = {}
    for k, v in t.items():
        if k == "q":
            sub[k] = v[b:b + 1, kvh * hq:(kvh + 1) * hq]
        elif k in ("seq_lens", "win_lens"):
            sub[k] = v[b:b + 1]
        else:
            sub[k] = v[b:b + 1, kvh:kvh + 1]
        sub[k] = sub[k].contiguous().cpu()
    w = inputs.Workload(wl.name, 1, hq, 1, [wl.lens[b]], bits=wl.bits, k_layout=wl.k_layout, v_layout=wl.v_layout,
                        group=wl.group, sm_scale=wl.sm_scale, window=wl.window)
    assert w.t_cap == wl.t_cap or w.t_cap <= wl.t_cap
    return sub, w


def sampled_parity(m, wl, units):
    t = inputs.generate(wl, "cuda")
    win = {}
    if "k_win" in t:
        win = dict(k_win=t["k_win"], v_win=t["v_win"], win_lens=t["win_lens"])
    out = m.decode_attn(t["q"], t["k_codes"], t["k_scale"], t["k_off"], t["v_codes"], t["v_scale"], t["v_off"],
                        t["seq_lens"], bits=wl.bits, k_layout=wl.k_layout, v_layout=wl.v_layout, group=wl.group,
                        **win)
    torch.cuda.synchronize()
    got_all = out.float().cpu().numpy().astype(np.float64)
    hq = wl.hq_per_kv
    worst = (0.0, 0.0)
    for b, kvh in units:
        sub, w = unit_slice(t, wl, b, kvh)
        x = to_oracle(sub, w)
        x.T_cap = wl.t_cap
        ref = oracle.decode_ref(x)[0]
        got = got_all[b, kvh * hq:(kvh + 1) * hq]
        mx, rl2 = assert_parity(got, ref, f"{wl.name} unit ({b},{kvh})")
        worst = (max(worst[0], mx), max(worst[1], rl2))
    del t
    torch.cuda.empty_cache()
    return worst


@pytest.mark.parametrize("batch,ctx", [(1, 131072), (8, 32768), (32, 32768), (64, 131072)])
def test_int2_full_size_sampled(lbkv, batch, ctx):
    """The INT2 token-wise decode shape at full size (batch 32 at 32K context is the
    benchmark's headline launch), on sampled (sequence, KV head) units."""
    wl = inputs.decode_int2(batch, ctx)
    sampled_parity(lbkv, wl, [(0, 0), (batch - 1, 7), (batch // 2, 3)])


@pytest.mark.parametrize("batch,ctx", [(1, 32768), (64, 131072)])
def test_int4_full_size_sampled(lbkv, batch, ctx):
    wl = inputs.decode_int4(batch, ctx)
    sampled_parity(lbkv, wl, [(0, 0), (batch - 1, 5)])


@pytest.mark.parametrize("bits,batch,ctx", [(2, 1, 4096), (2, 1, 16384), (2, 1, 32768), (2, 1, 65536), (2, 8, 16384),
                                            (4, 1, 16384), (4, 8, 4096), (4, 1, 131072)])
def test_few_pairs_every_unit(lbkv, bits, batch, ctx):
    """Few (sequence, KV head) pairs at full context: on a 152-SM GPU these shapes run as
    thread-block clusters, one per pair (2 to 8 CTAs that merge in distributed shared memory)
    or several per pair (batch 1 from 32K: four clusters of four, whose partials the last
    cluster merges); every unit is compared with the oracle."""
    wl = (inputs.decode_int2 if bits == 2 else inputs.decode_int4)(batch, ctx)
    sampled_parity(lbkv, wl, [(b, h) for b in range(batch) for h in range(wl.num_kv_heads)])


@pytest.mark.parametrize("lens,window", [([32768], 128), ([32000, 1999], 0), ([30000, 0, 12345], 64),
                                         ([65536, 17], 0)])
def test_few_pairs_ragged_and_window(lbkv, lens, window):
    """Few pairs with ragged lengths, an empty sequence or a bf16 window, in the cluster
    modes (clusters of one pair with fewer items than CTAs, the window merged by the last
    cluster of a pair); every unit is compared with the oracle."""
    wl = inputs.Workload(f"few-pairs-{len(lens)}", len(lens), 32, 8, lens, bits=2, group=128, s_range=(0.01, 0.1),
                         window=window, seed=11)
    sampled_parity(lbkv, wl, [(b, h) for b in range(len(lens)) for h in range(wl.num_kv_heads)])


@pytest.mark.parametrize("bits", [2, 4])
@pytest.mark.parametrize("kl,vl", [(1, 0), (0, 1)])
def test_mixed_layouts_ragged_sampled(lbkv, bits, kl, vl):
    """Batch 16, lengths uniform in [1K, 64K] and never a multiple of 128."""
    wl = inputs.mixed_layout(bits, kl, vl)
    sampled_parity(lbkv, wl, [(0, 0), (5, 4), (15, 7), (int(np.argmin(wl.lens)), 1)])


@pytest.mark.parametrize("g,hq", [(128, 4), (64, 2), (128, 8), (32, 1), (32, 8)])
def test_long_context_window_sampled(lbkv, g, hq):
    """100,000-token context: 99,872 INT2 tokens + a 128-token bf16 window."""
    wl = inputs.long_context(1, group=g, hq_per_kv=hq)
    sampled_parity(lbkv, wl, [(0, 0), (0, wl.num_kv_heads - 1)])


def test_bounded_wait_reports_and_the_context_survives(lbkv):
    """A wait that nothing completes gives up after its limit, records the timeout code in
    the status word and lets the warp go on; the context then still decodes correctly."""
    t0 = time.perf_counter()
    code, went_on = lbkv._binding.selftest_wait_timeout(20_000_000)  # 20 ms
    assert (code, went_on) == (1, 1)
    assert time.perf_counter() - t0 < 5.0
    check(lbkv, inputs.tiny_int2())



@pytest.mark.parametrize("bits,hq_total,hkv,ctx,kl,vl,g", [
    (2, 32, 4, 65536, 0, 0, 128),   # 8 queries per KV head (8-warp kernel)
    (4, 8, 8, 65536, 0, 0, 128),    # 1 query per KV head
    (2, 16, 8, 65536, 1, 1, 128),   # channel-wise K and V
    (2, 32, 8, 65536, 0, 0, 32),    # token-wise V with 4 channel groups (16 columns, 8 warps)
    (4, 32, 8, 49152, 0, 1, 64),
])
def test_few_pairs_other_shapes(lbkv, bits, hq_total, hkv, ctx, kl, vl, g):
    """Batch 1 at long context for other query ratios, layouts and groups (cluster modes with
    8-warp kernels and other column modes); every unit is compared with the oracle."""
    s = (0.01, 0.1) if bits == 2 else (0.002, 0.02)
    wl = inputs.Workload(f"few-pairs-hq{hq_total}-kv{hkv}", 1, hq_total, hkv, ctx - 77, bits=bits, k_layout=kl,
                         v_layout=vl, group=g, s_range=s, seed=12)
    sampled_parity(lbkv, wl, [(0, h) for h in range(hkv)])


@pytest.mark.parametrize("bits,batch,ctx,window,want", [
    (2, 32, 32768, False, (152, 0, 1)),   # the headline: the split-decode grid
    (2, 8, 32768, False, (128, 2, 1)),    # one cluster of 2 per pair
    (2, 1, 16384, False, (64, 8, 1)),     # one cluster of 8 per pair
    (2, 1, 32768, False, (128, 4, 4)),    # four clusters of 4 per pair
    (2, 1, 99968, True, (144, 2, 9)),     # long context with a window: nine clusters of 2
    (4, 1, 131072, False, (152, 0, 1)),   # INT4 batch 1 at 128K: the split-decode grid
])
def test_launch_modes_on_this_device(lbkv, bits, batch, ctx, window, want):
    """The launch each mode's parity tests rely on (on a 152-SM GB300; other devices may
    choose other shapes, which the parity tests cover as well)."""
    if torch.cuda.get_device_properties(0).multi_processor_count != 152:
        pytest.skip("launch shapes are stated for 152 SMs")
    info = lbkv.decode_launch_info(batch, 32, 8, ctx, bits, window=window)
    assert (info["grid"], info["cluster"], info["split"]) == want, info
