"""The benchmark's algorithmic bytes (the roofline's numerator) against per-token figures worked
out by hand from the cache layout (no GPU).

Per token and KV head, a side stores D·b/8 bytes of codes; a token-wise side adds one fp16 scale
and one fp16 offset per group of g channels (4·D/g bytes), a channel-wise side one pair per
channel per g tokens (4·D bytes per started group). Each call also reads Q, writes the output
(bf16 [B][Hq][D] each) and reads the int32 lengths; a bf16 window adds its K and V rows and its
lengths."""

import bench
from bit_kv_cache_split_gb300 import inputs


def test_headline_is_72_bytes_per_token_and_head():
    # INT2, g128, token-wise K and V: 2 x 32 B of codes + 2 x 4 B of scale/offset = 72 B
    wl = inputs.decode_int2(32, 32768)
    per_token = 72
    expected = 32 * 8 * 32768 * per_token + 2 * 32 * 32 * 128 * 2 + 4 * 32
    assert bench.algorithmic_bytes(wl) == expected == 604504192


def test_int4_is_136_bytes_per_token_and_head():
    wl = inputs.decode_int4(8, 4096)
    assert bench.algorithmic_bytes(wl) == 8 * 8 * 4096 * (2 * 64 + 8) + 2 * 8 * 32 * 128 * 2 + 4 * 8


def test_tokenwise_group_32_has_four_scale_pairs_per_token():
    wl = inputs.Workload("g32", 2, 8, 2, [100, 7], bits=2, group=32)
    per_token = 2 * 32 + 2 * 4 * 4  # codes, then 4 groups x (scale + offset) x 2 B per side
    assert bench.algorithmic_bytes(wl) == 2 * (100 + 7) * per_token + 2 * 2 * 8 * 128 * 2 + 4 * 2


def test_channelwise_side_counts_started_groups():
    # K channel-wise over 128-token groups: 300 tokens start 3 groups, 128 start 1, 129 start 2
    lens = [300, 128, 129]
    wl = inputs.Workload("cw", 3, 32, 8, lens, bits=2, k_layout=1, v_layout=0, group=128)
    per_head = sum(2 * 32 * L + 4 * L + 4 * 128 * -(-L // 128) for L in lens)
    assert bench.algorithmic_bytes(wl) == 8 * per_head + 2 * 3 * 32 * 128 * 2 + 4 * 3


def test_window_adds_its_rows_and_lengths():
    base = inputs.decode_int2(4, 4096)
    win = inputs.Workload(**{**base.__dict__, "window": 128})
    assert bench.algorithmic_bytes(win) - bench.algorithmic_bytes(base) == 4 * 8 * 128 * 128 * 2 * 2 + 4 * 4
