"""Test helpers: tensor <-> oracle marshalling and an independent numpy view
of the documented cache layout, used to build dense K/V for library routines.
"""

from __future__ import annotations

import os

import numpy as np
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def golden_lines(name):
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                yield line


def bits16(t: torch.Tensor) -> np.ndarray:
    """Raw 16-bit patterns of a bf16/fp16 tensor as uint16 numpy."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def to_oracle(t: dict, wl) -> oracle.DecodeInputs:
    """Marshal generated tensors into oracle inputs (host copies of every array)."""
    return oracle.inputs_from_tensors(t, bits=wl.bits, k_layout=wl.k_layout, v_layout=wl.v_layout, group=wl.group,
                                      Hkv=wl.num_kv_heads, T_cap=wl.t_cap, sm_scale=wl.sm_scale)


def np_unpack(codes: np.ndarray, bits: int) -> np.ndarray:
    """[..., D*bits/8] uint8 -> [..., D] int codes (code i of a byte in bits [b*i, b*i+b))."""
    per = 8 // bits
    parts = [(codes >> (bits * i)) & ((1 << bits) - 1) for i in range(per)]
    return np.stack(parts, axis=-1).reshape(*codes.shape[:-1], codes.shape[-1] * per).astype(np.int64)


def np_dequant(codes, scale, off, bits, layout, group):
    """Dense s*q + z in fp64 for [B][H][T][...] arrays (fp16 scale/off as float16 arrays)."""
    q = np_unpack(codes, bits).astype(np.float64)
    s = scale.astype(np.float64)
    z = off.astype(np.float64)
    if layout == oracle.TOKENWISE:
        s = np.repeat(s, group, axis=-1)
        z = np.repeat(z, group, axis=-1)
    else:
        s = np.repeat(s, group, axis=-2)
        z = np.repeat(z, group, axis=-2)
    return s * q + z


def sdpa_reference(q, k, v, lens, sm_scale=None):
    """Dense attention via torch's scaled_dot_product_attention in fp64.

    q [B][Hq][D], k/v [B][Hkv][T][D] (numpy fp64), lens [B]. GQA by repeating KV heads.
    """
    B, Hq, D = q.shape
    Hkv = k.shape[1]
    out = np.zeros((B, Hq, D))
    for b in range(B):
        L = int(lens[b])
        if L == 0:
            continue
        qt = torch.from_numpy(q[b]).reshape(1, Hq, 1, D)
        kt = torch.from_numpy(np.ascontiguousarray(k[b, :, :L])).repeat_interleave(Hq // Hkv, dim=0)[None]
        vt = torch.from_numpy(np.ascontiguousarray(v[b, :, :L])).repeat_interleave(Hq // Hkv, dim=0)[None]
        o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, scale=sm_scale)
        out[b] = o[0, :, 0].numpy()
    return out


def bf16_to_np(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().to(torch.float64).numpy()


def f16_to_np(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().numpy()
