"""Pins of the CPU oracle against values the pages print or that follow from
them by hand (fixtures under tests/golden/, each citing its source)."""

import numpy as np
import pytest

from tests.helpers import golden_lines


def test_unpack_bit_table(oracle_lib):
    """Hand-written bytes decode to the documented code order (golden/unpack_bits.txt)."""
    n = 0
    for line in golden_lines("unpack_bits.txt"):
        f = line.split()
        bits, byte, codes = int(f[0]), int(f[1], 16), [int(x) for x in f[2:]]
        row = np.array([byte], dtype=np.uint8)
        got = [oracle_lib.unpack_code(row, bits, d) for d in range(8 // bits)]
        assert got == codes, line
        n += 1
    assert n >= 8


def test_unpack_multibyte_rows(oracle_lib):
    """Code d lives in byte floor(d*b/8): a row of distinct bytes decodes position by position."""
    row = np.array([0xE4, 0x1B, 0xA5, 0x0F], dtype=np.uint8)
    assert [oracle_lib.unpack_code(row, 2, d) for d in range(16)] == [0, 1, 2, 3, 3, 2, 1, 0, 1, 1, 2, 2, 3, 3, 0, 0]
    assert [oracle_lib.unpack_code(row, 4, d) for d in range(8)] == [4, 14, 11, 1, 5, 10, 15, 0]


def _receipt():
    vals = {}
    for line in golden_lines("receipt.txt"):
        k, *rest = line.split()
        vals[k] = [float(x) for x in rest]
    return vals


def test_receipt_raw_and_quantity_sums(oracle_lib):
    """acc-fold with (s, z) = (1, 0) gives the raw subtotal, (0, 1) the quantity total."""
    r = _receipt()
    w, q = r["quantities"], [int(x) for x in r["stickers"]]
    assert oracle_lib.acc_fold(w, q, 1.0, 0.0) == r["raw_subtotal"][0] == 13
    assert oracle_lib.acc_fold(w, q, 0.0, 1.0) == r["quantity_total"][0] == 6


def test_receipt_fast_cashier_equals_slow_cashier(oracle_lib):
    """rate*13 + fee*6 equals converting every sticker first, exactly (binary fractions)."""
    r = _receipt()
    w, q = r["quantities"], [int(x) for x in r["stickers"]]
    rate, fee, total = r["rate_fee_total"]
    folded = oracle_lib.acc_fold(w, q, rate, fee)
    slow = oracle_lib.weighted_dequant_sum(w, q, [rate] * 3, [fee] * 3)
    assert folded == slow == total


def test_receipt_per_line_rate(oracle_lib):
    """With one rate per line the fast cashier pre-multiplies each quantity by its rate."""
    r = _receipt()
    w, q = r["quantities"], [int(x) for x in r["stickers"]]
    rates, fees = [0.5, 0.25, 2.0], [0.125, 0.125, 0.125]
    folded = oracle_lib.operand_fold(w, q, rates, fees)
    slow = oracle_lib.weighted_dequant_sum(w, q, rates, fees)
    # 3*(0.5*2) + 1*(0.25*1) + 2*(2*3) + 0.125*6 = 3 + 0.25 + 12 + 0.75 = 16
    assert folded == slow == 16.0


def test_fold_table(oracle_lib):
    """The oracle picks the fold the fold table names for each (side, layout)."""
    side = {"K": 0, "V": 1}
    layout = {"token": oracle_lib.TOKENWISE, "channel": oracle_lib.CHANNELWISE}
    fold = {"acc": oracle_lib.ACC_FOLD, "operand": oracle_lib.OPERAND_FOLD}
    rows = list(golden_lines("fold_table.txt"))
    assert len(rows) == 4
    for line in rows:
        s, lay, _prod, _axis, f = line.split()
        assert oracle_lib.fold_kind(side[s], layout[lay]) == fold[f], line


def _tiny_problem(oracle_lib, hq, g, bits, k_layout, v_layout, L, seed=0, D=128):
    rng = np.random.default_rng(seed)
    T = ((L + 127) // 128) * 128
    T = max(T, 128)
    B, Hkv = 1, 1
    row = D * bits // 8

    def sz(layout):
        shape = (B, Hkv, T, D // g) if layout == oracle_lib.TOKENWISE else (B, Hkv, T // g, D)
        s = rng.uniform(0.01, 0.1, shape).astype(np.float16).view(np.uint16)
        z = rng.uniform(-0.2, 0.2, shape).astype(np.float16).view(np.uint16)
        return s, z

    ks, kz = sz(k_layout)
    vs, vz = sz(v_layout)
    q = (rng.standard_normal((B, hq, D)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    return oracle_lib.DecodeInputs(
        q=q, k_codes=rng.integers(0, 256, (B, Hkv, T, row), dtype=np.uint8), k_scale=ks, k_off=kz,
        v_codes=rng.integers(0, 256, (B, Hkv, T, row), dtype=np.uint8), v_scale=vs, v_off=vz,
        seq_lens=[L], bits=bits, k_layout=k_layout, v_layout=v_layout, group=g, Hkv=Hkv, T_cap=T)


@pytest.mark.parametrize("layouts", [(0, 0), (1, 0), (0, 1), (1, 1)])
def test_op_count_closed_form(oracle_lib, layouts):
    """Folding costs 2*h_q/g scale/offset operations per stored value (golden/budget.txt)."""
    for line in golden_lines("budget.txt"):
        hq, g, want = line.split()
        hq, g, want = int(hq), int(g), float(want)
        x = _tiny_problem(oracle_lib, hq, g, 2, *layouts, L=256)
        _, ops, values = oracle_lib.decode_folded(x, block=128)
        assert ops / values == pytest.approx(want, rel=0, abs=1e-15), (line, layouts)
    # the pages' example: a 16x cut against one operation per value
    x = _tiny_problem(oracle_lib, 4, 128, 2, *layouts, L=256)
    _, ops, values = oracle_lib.decode_folded(x, block=128)
    assert values / ops == 16.0


def test_break_even(oracle_lib):
    """Folding beats per-value dequantization exactly when g > 2*h_q."""
    for hq, g in [(8, 16), (8, 32), (4, 8), (4, 16)]:
        if 128 % g:
            continue
        x = _tiny_problem(oracle_lib, hq, g, 2, 0, 0, L=128)
        _, ops, values = oracle_lib.decode_folded(x, block=128)
        assert (ops < values) == (g > 2 * hq), (hq, g, ops / values)


def test_pack_golden_cases(oracle_lib):
    """Hand-computed quantizer cases, token-wise and channel-wise (golden/pack_cases.txt)."""
    n = 0
    for line in golden_lines("pack_cases.txt"):
        bits, vals, s_hex, z_hex, codes = [p.strip() for p in line.split("|")]
        bits = int(bits)
        vals = np.array([float(v) for v in vals.split()], dtype=np.float32)
        codes = [int(c) for c in codes.split()]
        xb = (vals.view(np.uint32) >> 16).astype(np.uint16)
        assert np.all((xb.astype(np.uint32) << 16).view(np.float32) == vals), "fixture values must be bf16-exact"
        g = len(vals)
        # token-wise: one token, g channels
        x = xb.reshape(1, 1, 1, g)
        c, s, z = oracle_lib.pack(x, [1], bits, oracle_lib.TOKENWISE, g)
        got = [oracle_lib.unpack_code(c[0, 0, 0], bits, d) for d in range(g)]
        assert (int(s.ravel()[0]), int(z.ravel()[0]), got) == (int(s_hex, 16), int(z_hex, 16), codes), line
        # channel-wise: g tokens of one channel (every channel of the row identical)
        D = 8 // bits * 2
        x = np.repeat(xb.reshape(1, 1, g, 1), D, axis=3)
        c, s, z = oracle_lib.pack(x, [g], bits, oracle_lib.CHANNELWISE, g)
        got = [oracle_lib.unpack_code(c[0, 0, t], bits, 0) for t in range(g)]
        assert (int(s[0, 0, 0, 0]), int(z[0, 0, 0, 0]), got) == (int(s_hex, 16), int(z_hex, 16), codes), line
        n += 1
    assert n >= 6
