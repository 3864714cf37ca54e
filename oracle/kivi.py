"""KIVI asymmetric min/max quantisation and bit packing (CPU oracle).

Test infrastructure: see the package docstring for who may import this.

Sources (page title, section):
  * posttrainllm "StreamingLLM + KIVI" doc, "Affine quantisation formula":
    scale = max(eps, (xMax - xMin) / (qMax - qMin)), eps = 1e-5, zero = xMin,
    q = round((x - zero) / scale + qMin), x_dq = (q - qMin) * scale + zero.
  * same doc, "The bug class the previous attempt hit": the eps clamp (item 1),
    fp16 scales promoted to fp32 before dequantisation (item 2), a clamp range
    that reaches both end codes (item 3).
  * same doc, "Caveats": quantise per fixed-size token group and freeze the
    scales at the group boundary (the KIVI group idea), used here with
    32-token K groups and 32-channel V groups.
  * Foundry "TurboQuant KV Cache Compression - Spec", "Step 3: Packing":
    [v0:2][v1:2][v2:2][v3:2] and [v0:4][v1:4] per byte; 3-bit codes eight to
    three bytes (the page's no-waste form for the memory-bound case).

Readings where the pages leave a step open:
  * Codes are stored unsigned: q_u = q - qMin, so the qMin offset drops out
    and the code range is 0 .. 2^b - 1.
  * round() is round-half-to-even (numpy.rint).
  * The codes are computed from the STORED fp16 scale and zero, promoted to
    fp32, so quantise and dequantise use the same numbers.
  * The eps clamp is applied in fp32 before the fp16 rounding of the scale.
  * Packing puts v0 in the least-significant bits of each byte, and packs
    along the channel axis of one token row. 3-bit codes are packed tight:
    the row is one little-endian bit string with code i at bits 3i .. 3i+2
    (eight codes in three bytes), the page's no-waste form rather than its
    two-per-byte first cut, because the decode is memory-bound.
  * Every step is fp32 with each operation rounded on its own (numpy applies
    one ufunc at a time, so nothing is fused).
"""
from __future__ import annotations

import numpy as np

EPS = np.float32(1e-5)
GROUP = 32
FP16_MAX = 65504.0


def levels(bits: int) -> int:
    """Largest unsigned code, 2^b - 1 (qMax - qMin of the signed form)."""
    if bits not in (2, 3, 4, 8):
        raise ValueError(f"KIVI bit width must be 2, 3, 4 or 8, got {bits}")
    return (1 << bits) - 1


def _check_finite(x: np.ndarray) -> None:
    if not np.all(np.isfinite(x)):
        raise ValueError("NaN/Inf input: quantisation is undefined for it")
    if np.any(np.abs(x) > FP16_MAX):
        raise ValueError("input outside the fp16 range: the fp16 zero would overflow")


def quantize_slices(x: np.ndarray, bits: int):
    """Quantise each slice along the last axis with its own (scale, zero).

    x: float32 [..., n]. Returns (codes uint8 [..., n], scale fp16 [...],
    zero fp16 [...]).
    """
    x = np.asarray(x, dtype=np.float32)
    _check_finite(x)
    lb = np.float32(levels(bits))
    mn = x.min(axis=-1)
    mx = x.max(axis=-1)
    s32 = np.maximum((mx - mn) / lb, EPS)          # fp32 sub, fp32 div, eps clamp
    s_h = s32.astype(np.float16)                   # stored scale (RNE)
    z_h = mn.astype(np.float16)                    # stored zero (RNE)
    s = s_h.astype(np.float32)[..., None]
    z = z_h.astype(np.float32)[..., None]
    q = np.rint((x - z) / s)                       # fp32 sub, fp32 div, half-even
    q = np.clip(q, np.float32(0.0), lb)
    return q.astype(np.uint8), s_h, z_h


def dequantize_slices(codes: np.ndarray, s_h: np.ndarray, z_h: np.ndarray) -> np.ndarray:
    """x_dq = q * scale + zero in fp32, scale and zero promoted from fp16 first."""
    s = np.asarray(s_h, np.float16).astype(np.float32)[..., None]
    z = np.asarray(z_h, np.float16).astype(np.float32)[..., None]
    return codes.astype(np.float32) * s + z


def quantize_k_group(k_rows: np.ndarray, bits: int):
    """K of one 32-token group: one (scale, zero) per channel over the 32 tokens.

    k_rows: float32 [..., 32, D]. Returns codes uint8 [..., 32, D],
    scale/zero fp16 [..., D].
    """
    q, s, z = quantize_slices(np.swapaxes(k_rows, -1, -2), bits)
    return np.swapaxes(q, -1, -2), s, z


def dequantize_k_group(codes, s_h, z_h) -> np.ndarray:
    return np.swapaxes(dequantize_slices(np.swapaxes(codes, -1, -2), s_h, z_h), -1, -2)


def quantize_v_rows(v_rows: np.ndarray, bits: int):
    """V per token over 32-channel groups.

    v_rows: float32 [..., T, D]. Returns codes uint8 [..., T, D] and
    scale/zero fp16 [..., T, D/32].
    """
    *lead, T, D = v_rows.shape
    q, s, z = quantize_slices(v_rows.reshape(*lead, T, D // GROUP, GROUP), bits)
    return q.reshape(*lead, T, D), s, z


def quantize_slices_q4_0(x: np.ndarray):
    """The symmetric 4-bit block format P3 names for V ("`--kv q2k`": "V at 4
    bits per token (q4_0)"), as its public definition has it: per slice of 32,
    m = the value of largest magnitude (the first on ties), d = m / -8, code
    q = min(15, floor(x / d + 8.5)) and value (q - 8) d. Written in the affine
    form of this cache: scale d, zero -8 d (exact in fp16). Readings: d is
    stored in fp16 and the codes use the stored value, like KIVI's; a slice
    of zeros has d = 0 and every code 8.

    x: float32 [..., n]. Returns (codes uint8 [..., n], scale fp16 [...],
    zero fp16 [...]).
    """
    x = np.asarray(x, np.float32)
    _check_finite(x)
    idx = np.argmax(np.abs(x), axis=-1)                      # first index of the largest |x|
    m = np.take_along_axis(x, idx[..., None], axis=-1)[..., 0]
    d_h = (m / np.float32(-8.0)).astype(np.float16)           # fp32 division, stored fp16
    z_h = (d_h.astype(np.float32) * np.float32(-8.0)).astype(np.float16)
    d = d_h.astype(np.float32)[..., None]
    with np.errstate(divide="ignore", invalid="ignore"):
        t = np.floor((x / d) + np.float32(8.5))               # fp32 divide, fp32 add
    q = np.where(d == 0, np.float32(8.0), np.clip(t, np.float32(0.0), np.float32(15.0)))
    return q.astype(np.uint8), d_h, z_h


def quantize_v_rows_q4_0(v_rows: np.ndarray):
    """V per token over 32-channel groups in the symmetric q4_0 form."""
    *lead, T, D = v_rows.shape
    q, s, z = quantize_slices_q4_0(v_rows.reshape(*lead, T, D // GROUP, GROUP))
    return q.reshape(*lead, T, D), s, z


def dequantize_v_rows(codes, s_h, z_h) -> np.ndarray:
    *lead, T, D = codes.shape
    x = dequantize_slices(codes.reshape(*lead, T, D // GROUP, GROUP), s_h, z_h)
    return x.reshape(*lead, T, D)


def pack_codes(codes: np.ndarray, bits: int) -> np.ndarray:
    """Pack codes along the last axis, v0 in the least-significant bits
    (Foundry spec, "Step 3: Packing": 2-bit [v0:2][v1:2][v2:2][v3:2], 4-bit
    [v0:4][v1:4], 8-bit one code per byte; 3-bit eight codes in three bytes,
    code i at bits 3i .. 3i+2 of the row's little-endian bit string).

    codes: uint8 [..., D] with values < 2^bits. Returns uint8 [..., D * bits / 8].
    """
    D = codes.shape[-1]
    if (D * bits) % 8 or (bits == 3 and D % 8):
        raise ValueError("row length must fill whole bytes")
    if bits == 3:
        c = codes.reshape(*codes.shape[:-1], D // 8, 8).astype(np.uint32)
        word = np.zeros(c.shape[:-1], np.uint32)            # 24 bits per eight codes
        for i in range(8):
            word |= c[..., i] << np.uint32(3 * i)
        out = np.stack([(word >> np.uint32(8 * k)) & np.uint32(0xFF) for k in range(3)], axis=-1)
        return out.reshape(*codes.shape[:-1], D * 3 // 8).astype(np.uint8)
    per = 8 // bits
    c = codes.reshape(*codes.shape[:-1], D // per, per).astype(np.uint16)
    out = np.zeros(c.shape[:-1], np.uint16)
    for i in range(per):
        out |= c[..., i] << (i * bits)
    return out.astype(np.uint8)


def unpack_codes(packed: np.ndarray, bits: int) -> np.ndarray:
    """Inverse of pack_codes."""
    if bits == 3:
        p = packed.reshape(*packed.shape[:-1], packed.shape[-1] // 3, 3).astype(np.uint32)
        word = p[..., 0] | (p[..., 1] << np.uint32(8)) | (p[..., 2] << np.uint32(16))
        c = np.stack([(word >> np.uint32(3 * i)) & np.uint32(7) for i in range(8)], axis=-1)
        return c.reshape(*packed.shape[:-1], packed.shape[-1] * 8 // 3).astype(np.uint8)
    per = 8 // bits
    mask = (1 << bits) - 1
    p = packed.astype(np.uint16)[..., None]
    shifts = (np.arange(per, dtype=np.uint16) * bits)
    c = (p >> shifts) & mask
    return c.reshape(*packed.shape[:-1], packed.shape[-1] * per).astype(np.uint8)
