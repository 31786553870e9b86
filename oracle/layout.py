"""Byte layout of FP8 and TQ3 pages, written from the format spec in
``include/mkv.h`` (section "Storage formats").  Independent of the CUDA
implementation; the GPU parity tests compare exported page bytes with what
this module packs.

One page holds ``P`` tokens of one layer (P a multiple of 64).  For each kv
head h (in order) the page stores a K plane then a V plane; a plane is the
code bytes followed by ``P`` little-endian fp16 scales (token order).

FP8 (1 byte per element):
  K codes: 64-token blocks, each stored as D/16 columns of 16 bytes:
           byte ``(t//64)*64*D + (j//16)*1024 + (t%64)*16 + j%16``.
  V codes: 8-token groups, each dimension's 8 bytes together:
           byte ``(t//8)*8*D + j*8 + t%8``.

TQ3 (3 bits per element): codes are grouped in 12-byte units of 32 codes
(3 bits per code; no unit boundary falls inside a byte).  A unit is three
little-endian 32-bit words W0..W2:
  bits [4i, 4i+3) of W_k hold code (8k + i)          for i = 0..7, k = 0..2;
  bit  4i+3       of W_k holds bit k of code (24 + i).
  K codes: unit ``t*(D/32) + j//32``, code index ``j % 32``   (rows in order).
  V codes: unit ``j*(P/32) + t//32``, code index ``t % 32``
           (dimension-major: each dimension's codes in token order).
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
    """V plane codes [P, D] -> unit-ordered [D*P/32, 32]: unit j*(P/32) + t//32, code t%32."""
    P, D = codes.shape
    return np.ascontiguousarray(codes.T).reshape(D * (P // 32), 32)


def _tq3_v_from_units(units: np.ndarray, P: int, D: int) -> np.ndarray:
    return units.reshape(D, P).T.copy()


def _fp8_k_order(codes: np.ndarray) -> np.ndarray:
    """K plane codes [P, D] -> plane bytes: 64-token blocks of D/16 16-byte columns."""
    P, D = codes.shape
    blk = codes.reshape(P // 64, 64, D // 16, 16)          # [block, t%64, column, j%16]
    return blk.transpose(0, 2, 1, 3).reshape(-1)


def _fp8_k_from_bytes(b: np.ndarray, P: int, D: int) -> np.ndarray:
    blk = np.asarray(b).reshape(P // 64, D // 16, 64, 16)  # [block, column, t%64, j%16]
    return blk.transpose(0, 2, 1, 3).reshape(P, D)


def _fp8_v_order(codes: np.ndarray) -> np.ndarray:
    """V plane codes [P, D] -> plane bytes: 8-token groups, each dimension's 8 bytes together."""
    P, D = codes.shape
    grp = codes.reshape(P // 8, 8, D)                      # [group, t%8, j]
    return grp.transpose(0, 2, 1).reshape(-1)


def _fp8_v_from_bytes(b: np.ndarray, P: int, D: int) -> np.ndarray:
    grp = np.asarray(b).reshape(P // 8, D, 8)              # [group, j, t%8]
    return grp.transpose(0, 2, 1).reshape(P, D)


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
    assert P % 64 == 0 and D % 16 == 0
    plane = fp8_plane_bytes(P, D)
    out = np.zeros(fp8_page_bytes(P, Hkv, D), dtype=np.uint8)
    for h in range(Hkv):
        base = h * 2 * plane
        out[base: base + P * D] = _fp8_k_order(kc[:, h, :])
        out[base + P * D: base + plane] = _scales_bytes(ks[:, h])
        vb = base + plane
        out[vb: vb + P * D] = _fp8_v_order(vc[:, h, :])
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
        kc[:, h, :] = _fp8_k_from_bytes(page[base: base + P * D], P, D)
        ks[:, h] = _scales_from_bytes(page[base + P * D: base + plane])
        vb = base + plane
        vc[:, h, :] = _fp8_v_from_bytes(page[vb: vb + P * D], P, D)
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
