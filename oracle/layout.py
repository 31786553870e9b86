"""Byte layout of FP8 and TQ3 pages, written from the format spec in
``include/mkv.h`` (section "Storage formats").  Independent of the CUDA
implementation; the GPU parity tests compare exported page bytes with what
this module packs.

One page holds ``P`` tokens of one layer.  For each kv head h (in order) the
page stores a K plane then a V plane; a plane is the code bytes followed by
``P`` little-endian fp16 scales (token order).

FP8 (1 byte per element):
  K codes: row-major, byte ``t*D + j`` for token t, dim j.
  V codes: tokens paired (2v, 2v+1): byte ``v*2D + 2j + (t % 2)``, i.e. the two
           rows of a pair interleaved element by element.

TQ3 (3 bits per element): codes are grouped in 12-byte units of 32 codes
(3 bits per code, 32 codes per 12 bytes).  A unit is three little-endian
32-bit words W0..W2:
  bits [4i, 4i+3) of W_k hold code (8k + i)          for i = 0..7, k = 0..2;
  bit  4i+3       of W_k holds bit k of code (24 + i).
  K codes: unit ``t*(D/32) + j//32``, code index ``j % 32``   (rows in order).
  V codes: unit ``(t//2)*(D/16) + j//16``, code index ``2*(j % 16) + t % 2``
           (the two rows of a token pair interleaved code by code).
"""
from __future__ import annotations

import numpy as np


def fp8_plane_bytes(P: int, D: int) -> int:
    return P * D + 2 * P


def tq3_plane_bytes(P: int, D: int) -> int:
    return P * (3 * D // 8) + 2 * P


def fp8_page_bytes(P: int, Hkv: int, D: int) -> int:
    return Hkv * 2 * fp8_plane_bytes(P, D)


def tq3_page_bytes(P: int, Hkv: int, D: int) -> int:
    return Hkv * 2 * tq3_plane_bytes(P, D)


# ----------------------------------------------------------------- TQ3 units
def pack_units(codes32: np.ndarray) -> np.ndarray:
    """codes (..., 32) uint8 in 0..7 -> words (..., 3) uint32."""
    c = np.asarray(codes32, dtype=np.uint32)
    words = np.zeros(c.shape[:-1] + (3,), dtype=np.uint32)
    for k in range(3):
        w = np.zeros(c.shape[:-1], dtype=np.uint32)
        for i in range(8):
            w |= (c[..., 8 * k + i] & 7) << np.uint32(4 * i)
            w |= ((c[..., 24 + i] >> np.uint32(k)) & 1) << np.uint32(4 * i + 3)
        words[..., k] = w
    return words


def unpack_units(words: np.ndarray) -> np.ndarray:
    """words (..., 3) uint32 -> codes (..., 32) uint8."""
    w = np.asarray(words, dtype=np.uint32)
    codes = np.zeros(w.shape[:-1] + (32,), dtype=np.uint8)
    for k in range(3):
        for i in range(8):
            codes[..., 8 * k + i] = (w[..., k] >> np.uint32(4 * i)) & 7
    for i in range(8):
        v = np.zeros(w.shape[:-1], dtype=np.uint32)
        for k in range(3):
            v |= ((w[..., k] >> np.uint32(4 * i + 3)) & 1) << np.uint32(k)
        codes[..., 24 + i] = v
    return codes


def _tq3_k_unit_order(codes: np.ndarray) -> np.ndarray:
    """K plane codes [P, D] -> unit-ordered [P*D/32, 32]."""
    P, D = codes.shape
    return codes.reshape(P, D // 32, 32).reshape(P * D // 32, 32)


def _tq3_v_unit_order(codes: np.ndarray) -> np.ndarray:
    """V plane codes [P, D] -> unit-ordered [(P/2)*(D/16), 32], code index 2*(j%16)+parity."""
    P, D = codes.shape
    pair = codes.reshape(P // 2, 2, D // 16, 16)           # [v, parity, unit, j%16]
    unit = pair.transpose(0, 2, 3, 1)                      # [v, unit, j%16, parity]
    return unit.reshape((P // 2) * (D // 16), 32)


def _tq3_v_from_units(units: np.ndarray, P: int, D: int) -> np.ndarray:
    u = units.reshape(P // 2, D // 16, 16, 2).transpose(0, 3, 1, 2)
    return u.reshape(P, D)


def _scales_bytes(scales: np.ndarray) -> np.ndarray:
    return np.asarray(scales, dtype=np.float64).astype(np.float16).view(np.uint8)


def _scales_from_bytes(b: np.ndarray) -> np.ndarray:
    return np.frombuffer(np.ascontiguousarray(b).tobytes(), dtype=np.float16).astype(np.float64)


# ----------------------------------------------------------------- pages
def pack_fp8_page(kc, ks, vc, vs) -> np.ndarray:
    """kc/vc: uint8 [P, Hkv, D]; ks/vs: fp16 values [P, Hkv]. Returns page bytes."""
    kc = np.asarray(kc, dtype=np.uint8)
    vc = np.asarray(vc, dtype=np.uint8)
    P, Hkv, D = kc.shape
    plane = fp8_plane_bytes(P, D)
    out = np.zeros(fp8_page_bytes(P, Hkv, D), dtype=np.uint8)
    for h in range(Hkv):
        base = h * 2 * plane
        out[base: base + P * D] = kc[:, h, :].reshape(-1)
        out[base + P * D: base + plane] = _scales_bytes(ks[:, h])
        vb = base + plane
        pair = vc[:, h, :].reshape(P // 2, 2, D).transpose(0, 2, 1)   # [v, j, parity]
        out[vb: vb + P * D] = pair.reshape(-1)
        out[vb + P * D: vb + plane] = _scales_bytes(vs[:, h])
    return out


def unpack_fp8_page(page: np.ndarray, P: int, Hkv: int, D: int):
    page = np.asarray(page, dtype=np.uint8)
    plane = fp8_plane_bytes(P, D)
    kc = np.zeros((P, Hkv, D), dtype=np.uint8)
    vc = np.zeros((P, Hkv, D), dtype=np.uint8)
    ks = np.zeros((P, Hkv))
    vs = np.zeros((P, Hkv))
    for h in range(Hkv):
        base = h * 2 * plane
        kc[:, h, :] = page[base: base + P * D].reshape(P, D)
        ks[:, h] = _scales_from_bytes(page[base + P * D: base + plane])
        vb = base + plane
        vc[:, h, :] = page[vb: vb + P * D].reshape(P // 2, D, 2).transpose(0, 2, 1).reshape(P, D)
        vs[:, h] = _scales_from_bytes(page[vb + P * D: vb + plane])
    return kc, ks, vc, vs


def pack_tq3_page(kc, ks, vc, vs) -> np.ndarray:
    kc = np.asarray(kc, dtype=np.uint8)
    vc = np.asarray(vc, dtype=np.uint8)
    P, Hkv, D = kc.shape
    plane = tq3_plane_bytes(P, D)
    cb = P * (3 * D // 8)
    out = np.zeros(tq3_page_bytes(P, Hkv, D), dtype=np.uint8)
    for h in range(Hkv):
        base = h * 2 * plane
        out[base: base + cb] = pack_units(_tq3_k_unit_order(kc[:, h, :])).view(np.uint8).reshape(-1)
        out[base + cb: base + plane] = _scales_bytes(ks[:, h])
        vb = base + plane
        out[vb: vb + cb] = pack_units(_tq3_v_unit_order(vc[:, h, :])).view(np.uint8).reshape(-1)
        out[vb + cb: vb + plane] = _scales_bytes(vs[:, h])
    return out


def unpack_tq3_page(page: np.ndarray, P: int, Hkv: int, D: int):
    page = np.asarray(page, dtype=np.uint8)
    plane = tq3_plane_bytes(P, D)
    cb = P * (3 * D // 8)
    kc = np.zeros((P, Hkv, D), dtype=np.uint8)
    vc = np.zeros((P, Hkv, D), dtype=np.uint8)
    ks = np.zeros((P, Hkv))
    vs = np.zeros((P, Hkv))
    for h in range(Hkv):
        base = h * 2 * plane
        kw = np.ascontiguousarray(page[base: base + cb]).view(np.uint32).reshape(-1, 3)
        kc[:, h, :] = unpack_units(kw).reshape(P, D)
        ks[:, h] = _scales_from_bytes(page[base + cb: base + plane])
        vb = base + plane
        vw = np.ascontiguousarray(page[vb: vb + cb]).view(np.uint32).reshape(-1, 3)
        vc[:, h, :] = _tq3_v_from_units(unpack_units(vw), P, D)
        vs[:, h] = _scales_from_bytes(page[vb + cb: vb + plane])
    return kc, ks, vc, vs
