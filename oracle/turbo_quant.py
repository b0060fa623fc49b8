"""O3: compressed KV rows (TurboQuant: PolarQuant + QJL) and attention over them.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

Source: dendrite demo.tape, section "TurboQuant": the cache ships a KV
compression named "TurboQuant (PolarQuant + QJL)", tested for its
compression ratio, for the zero bias of the QJL estimate and for the
PolarQuant reconstruction error against fp16; it measures 3.05x at head_dim
128.  The pages give no algorithm, so the steps follow the published methods
they name:

* PolarQuant (Han, Kacham, Karbasi, Mirrokni, Zandieh, 2025): randomly
  precondition the vector, then apply the recursive polar transform -- level
  1 turns coordinate pairs into (radius, angle in [0, 2 pi)), every later
  level turns pairs of radii into (radius, angle in [0, pi/2]) -- until one
  radius (the norm) is left; quantize the angles, keep the norm.
* QJL (Zandieh, Daliri, Han, 2024): for a random Gaussian matrix S (m x d)
  keep sign(S e) and |e|; then for any q, sqrt(pi/2)/m * |e| * <S q, sign(S e)>
  is an unbiased estimate of <q, e>.
* TurboQuant (Zandieh, Daliri, Hadian, Mirrokni, 2025): an inner-product
  quantizer is an MSE quantizer plus a one-bit QJL sketch of its residual.

Readings (where the pages are silent):

* Keys use PolarQuant plus a QJL sketch of the key's residual (scores are
  inner products); values use PolarQuant alone (they are reconstructed).
* Preconditioning is the rotation R x = H (s * x) / sqrt(d): H the d x d
  Walsh-Hadamard matrix (Sylvester order), s a vector of random signs.  R is
  orthogonal, so <q, k> = <R q, R k> and attention can run in the rotated
  space, the output being rotated back with R^T.
* Level-1 angles take 4 bits (16 equal bins of [0, 2 pi): after a random
  rotation they are uniform).  The angle of level l >= 2 lies between the
  norms of two halves of k = 2^(l-1) coordinates each; for Gaussian-like
  rows its density is proportional to sin(2 phi)^(k-1), centred on pi/4 with
  a standard deviation close to 0.5 / sqrt(k - 1).  Those angles take 3 bits:
  8 equal bins of [pi/4 - w, pi/4 + w], w = min(pi/4, 1.6 / sqrt(k - 1))
  (3.2 standard deviations), angles beyond it falling into the end bins.  A
  code decodes to its bin's centre.  The norm is kept in fp32.  The QJL
  sketch has m = 128 sign bits and the residual norm in fp32.
* Records: a value row is 64 bytes, a key row 96 bytes (layout in
  ``pack_value`` / ``pack_key``); K + V take 160 bytes per row and head
  instead of 512 in bf16, 3.2x (the pages measure 3.05x with their own bit
  widths, which they do not state).
* The encoder takes its decisions (bins, signs) in fp32, one IEEE operation at
  a time in the order written below (no fused multiply-add), so the codes are
  a function of the input bits; everything the decoder and attention compute
  from the codes is evaluated in fp64.
"""
from __future__ import annotations

import math

import numpy as np

__all__ = ["D", "LEVELS", "M_QJL", "VALUE_BYTES", "KEY_BYTES", "upper_range", "rotate32", "rotate64", "unrotate64",
           "polar_encode32", "polar_decode32", "polar_decode64", "qjl_encode32", "qjl_estimate",
           "encode_value", "encode_key", "pack_value", "pack_key", "unpack_value", "unpack_key",
           "decode_value64", "decode_key64", "compressed_scores", "attention_compressed",
           "compression_ratio"]

D = 128
LEVELS = 7                  # log2(D)
M_QJL = 128
VALUE_BYTES = 64
KEY_BYTES = 96
F32 = np.float32

# bin boundaries and centres, each side of the comparison an fp32 number
_T1 = F32(math.tan(math.pi / 8))          # level 1: boundaries pi/8, pi/4, 3 pi/8 within a quadrant
_T3 = F32(math.tan(3 * math.pi / 8))
_INV_SQRT_D = F32(1.0 / math.sqrt(D))


def _level1_center(code):
    return (np.asarray(code, dtype=np.float64) + 0.5) * (math.pi / 8)


def upper_range(level: int):
    """(lo, hi) of the binned angle range of polar level ``level`` >= 2."""
    k = 2 ** (level - 1)
    w = min(math.pi / 4, 1.6 / math.sqrt(k - 1))
    return math.pi / 4 - w, math.pi / 4 + w


def _upper_tangents(level: int):
    """fp32 tangents of the 7 inner bin boundaries of a level >= 2."""
    lo, hi = upper_range(level)
    return [F32(math.tan(lo + j * (hi - lo) / 8)) for j in range(1, 8)]


def _upper_centers(level: int) -> np.ndarray:
    lo, hi = upper_range(level)
    return lo + (np.arange(8) + 0.5) * (hi - lo) / 8


# ----------------------------------------------------------------- rotation
def _fwht32(y: np.ndarray) -> np.ndarray:
    """In-place fast Walsh-Hadamard transform along the last axis in fp32:
    for h = 1, 2, 4, ..., pairs (i, i + h) with i & h == 0 become (u + v, u - v)."""
    y = y.astype(F32, copy=True)
    n = y.shape[-1]
    h = 1
    while h < n:
        v = y.reshape(y.shape[:-1] + (n // (2 * h), 2, h))
        a = v[..., 0, :].copy()
        b = v[..., 1, :].copy()
        v[..., 0, :] = a + b
        v[..., 1, :] = a - b
        h *= 2
    return y


def rotate32(x: np.ndarray, signs: np.ndarray) -> np.ndarray:
    """R x in fp32: sign flips, the butterflies, then one multiply by fp32(1/sqrt(d))."""
    y = np.asarray(x, dtype=F32) * np.asarray(signs, dtype=F32)
    return (_fwht32(y) * _INV_SQRT_D).astype(F32)


def _hadamard64(n: int) -> np.ndarray:
    H = np.array([[1.0]])
    while H.shape[0] < n:
        H = np.block([[H, H], [H, -H]])
    return H


def rotate64(x: np.ndarray, signs: np.ndarray) -> np.ndarray:
    """R x in fp64 (the definition: H (s * x) / sqrt(d))."""
    H = _hadamard64(D)
    return (np.asarray(x, np.float64) * np.asarray(signs, np.float64)) @ H.T / math.sqrt(D)


def unrotate64(y: np.ndarray, signs: np.ndarray) -> np.ndarray:
    """R^T y = s * (H y) / sqrt(d) (H is symmetric)."""
    H = _hadamard64(D)
    return (np.asarray(y, np.float64) @ H.T / math.sqrt(D)) * np.asarray(signs, np.float64)


# ------------------------------------------------------------ polar encoding
def _bin1(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """Level-1 code of the angle of (a, b) in [0, 2 pi): quadrant (0..3), the
    pair turned into the first quadrant, then its sub-bin from three fp32
    comparisons; (0, 0) codes 0."""
    q = np.where((a > 0) & (b >= 0), 0, np.where((a <= 0) & (b > 0), 1, np.where((a < 0) & (b <= 0), 2, 3)))
    x = np.where(q == 0, a, np.where(q == 1, b, np.where(q == 2, -a, -b))).astype(F32)
    y = np.where(q == 0, b, np.where(q == 1, -a, np.where(q == 2, -b, a))).astype(F32)
    sub = (y >= (x * _T1).astype(F32)).astype(np.int64) + (y >= x).astype(np.int64) + \
        (y >= (x * _T3).astype(F32)).astype(np.int64)
    code = 4 * q + sub
    return np.where((a == 0) & (b == 0), 0, code)


def _bin2(a: np.ndarray, b: np.ndarray, level: int) -> np.ndarray:
    """Code of the angle of (a, b), a, b >= 0, at polar level ``level``: the
    number of the level's 7 inner bin boundaries it reaches, each test
    b >= a * tan(boundary) in fp32; (0, 0) codes 0."""
    code = np.zeros(np.broadcast(a, b).shape, dtype=np.int64)
    for t in _upper_tangents(level):
        code += (b >= (a * t).astype(F32)).astype(np.int64)
    return np.where((a == 0) & (b == 0), 0, code)


def _radius32(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    aa = (a * a).astype(F32)
    bb = (b * b).astype(F32)
    return np.sqrt((aa + bb).astype(F32)).astype(F32)


def polar_encode32(x: np.ndarray):
    """PolarQuant codes of rotated rows ``x`` ``[..., 128]`` (fp32): returns
    (norm fp32 [...], level-1 codes [..., 64], codes of levels 2..7 [..., 63]
    in level order)."""
    x = np.asarray(x, dtype=F32)
    a, b = x[..., 0::2], x[..., 1::2]
    c1 = _bin1(a, b)
    r = _radius32(a, b)
    upper = []
    for level in range(2, LEVELS + 1):
        a, b = r[..., 0::2], r[..., 1::2]
        upper.append(_bin2(a, b, level))
        r = _radius32(a, b)
    return r[..., 0], c1, np.concatenate(upper, axis=-1)


def _decode(norm, c1, cu, cos1, sin1, cos2, sin2, mul):
    """The polar transform run backwards from the norm: level 7 down to 2 split
    a radius r into (r cos phi, r sin phi), level 1 into the coordinate pair.
    cos2 / sin2 [6][8]: the centres of levels 2..7."""
    r = np.asarray(norm)[..., None]
    sizes = [2 ** (LEVELS - l) for l in range(2, LEVELS + 1)]     # 32, 16, ..., 1
    offs = np.cumsum([0] + sizes)
    for lvl in range(LEVELS, 1, -1):                              # 7 .. 2
        k = lvl - 2
        code = cu[..., offs[k]:offs[k] + sizes[k]]
        lo, hi = mul(r, cos2[k][code]), mul(r, sin2[k][code])
        r = np.stack([lo, hi], axis=-1).reshape(lo.shape[:-1] + (2 * lo.shape[-1],))
    a, b = mul(r, cos1[c1]), mul(r, sin1[c1])
    return np.stack([a, b], axis=-1).reshape(a.shape[:-1] + (D,))


def polar_decode32(norm, c1, cu) -> np.ndarray:
    """Reconstruction in fp32, every product rounded (the encoder's residual)."""
    cos1 = np.cos(_level1_center(np.arange(16))).astype(F32)
    sin1 = np.sin(_level1_center(np.arange(16))).astype(F32)
    cen = np.stack([_upper_centers(l) for l in range(2, LEVELS + 1)])
    cos2, sin2 = np.cos(cen).astype(F32), np.sin(cen).astype(F32)
    return _decode(np.asarray(norm, F32), c1, cu, cos1, sin1, cos2, sin2, lambda u, v: (u * v).astype(F32))


def polar_decode64(norm, c1, cu) -> np.ndarray:
    """Reconstruction in fp64 from the bin centres."""
    t1 = _level1_center(np.arange(16))
    cen = np.stack([_upper_centers(l) for l in range(2, LEVELS + 1)])
    return _decode(np.asarray(norm, np.float64), c1, cu, np.cos(t1), np.sin(t1), np.cos(cen), np.sin(cen),
                   lambda u, v: u * v)


# ---------------------------------------------------------------------- QJL
def qjl_encode32(e: np.ndarray, S: np.ndarray):
    """QJL sketch of residual rows ``e`` ``[..., 128]`` (fp32) with ``S``
    ``[m][128]`` (fp32): bits [..., m] (1 where (S e)_j >= 0; each dot product
    summed in index order, product and sum rounded to fp32 in turn) and the
    residual norm (squares summed in index order, fp32)."""
    e = np.asarray(e, dtype=F32)
    S = np.asarray(S, dtype=F32)
    z = np.zeros(e.shape[:-1] + (S.shape[0],), dtype=F32)
    for i in range(e.shape[-1]):
        z = (z + (e[..., i:i + 1] * S[:, i]).astype(F32)).astype(F32)
    n2 = np.zeros(e.shape[:-1], dtype=F32)
    for i in range(e.shape[-1]):
        n2 = (n2 + (e[..., i] * e[..., i]).astype(F32)).astype(F32)
    return (z >= 0).astype(np.uint8), np.sqrt(n2).astype(F32)


def qjl_estimate(q: np.ndarray, bits: np.ndarray, enorm, S: np.ndarray) -> np.ndarray:
    """sqrt(pi/2)/m * |e| * <S q, sign(S e)> in fp64 (q [..., 128], bits [..., m])."""
    m = S.shape[0]
    sq = np.asarray(q, np.float64) @ np.asarray(S, np.float64).T
    sg = 2.0 * np.asarray(bits, np.float64) - 1.0
    return math.sqrt(math.pi / 2) / m * np.asarray(enorm, np.float64) * np.sum(sq * sg, axis=-1)


# ------------------------------------------------------------------- records
def encode_value(v, signs):
    """Rotated, polar-coded value rows: (norm, c1, cu)."""
    return polar_encode32(rotate32(v, signs))


def encode_key(k, signs, S):
    """Rotated, polar-coded key rows plus the QJL sketch of their fp32 residual:
    (norm, c1, cu, bits, residual norm)."""
    x = rotate32(k, signs)
    norm, c1, cu = polar_encode32(x)
    e = (x - polar_decode32(norm, c1, cu)).astype(F32)
    bits, enorm = qjl_encode32(e, S)
    return norm, c1, cu, bits, enorm


def _pack_polar(norm, c1, cu, nbytes):
    rows = np.asarray(norm).shape
    out = np.zeros(rows + (nbytes,), dtype=np.uint8)
    out[..., 0:4] = np.asarray(norm, F32)[..., None].view(np.uint8).reshape(rows + (4,))
    c1 = np.asarray(c1, np.uint8)
    out[..., 4:36] = (c1[..., 0::2] & 15) | ((c1[..., 1::2] & 15) << 4)
    # 63 codes of 3 bits, code i at bits [3 i, 3 i + 3) of a little-endian stream
    bits = np.zeros(rows + (24 * 8,), dtype=np.uint8)
    for k in range(3):
        bits[..., k:189:3] = (np.asarray(cu) >> k) & 1
    out[..., 36:60] = np.packbits(bits.reshape(rows + (24, 8)), axis=-1, bitorder="little")[..., 0]
    return out


def pack_value(norm, c1, cu):
    """Value record (64 bytes): [0, 4) norm fp32; [4, 36) 64 level-1 codes,
    4 bits each, code i in byte 4 + i / 2 (low nibble for even i); [36, 60)
    63 codes of levels 2..7 (level order), 3 bits each, code i at bit 3 i of a
    little-endian bit stream; [60, 64) zero."""
    return _pack_polar(norm, c1, cu, VALUE_BYTES)


def pack_key(norm, c1, cu, bits, enorm):
    """Key record (96 bytes): [0, 64) as a value record; [64, 80) the 128 QJL
    bits, bit j in byte 64 + j / 8 at bit j % 8; [80, 84) residual norm fp32;
    [84, 96) zero."""
    out = _pack_polar(norm, c1, cu, KEY_BYTES)
    rows = np.asarray(norm).shape
    out[..., 64:80] = np.packbits(np.asarray(bits, np.uint8).reshape(rows + (16, 8)), axis=-1,
                                  bitorder="little")[..., 0]
    out[..., 80:84] = np.asarray(enorm, F32)[..., None].view(np.uint8).reshape(rows + (4,))
    return out


def _unpack_polar(rec):
    rec = np.asarray(rec, np.uint8)
    rows = rec.shape[:-1]
    norm = rec[..., 0:4].copy().view(F32).reshape(rows)
    lo, hi = rec[..., 4:36] & 15, rec[..., 4:36] >> 4
    c1 = np.stack([lo, hi], axis=-1).reshape(rows + (64,)).astype(np.int64)
    bits = np.unpackbits(rec[..., 36:60][..., None], axis=-1, bitorder="little").reshape(rows + (192,))
    cu = bits[..., 0:189:3].astype(np.int64) + 2 * bits[..., 1:189:3] + 4 * bits[..., 2:189:3]
    return norm, c1, cu


def unpack_value(rec):
    return _unpack_polar(rec)


def unpack_key(rec):
    rec = np.asarray(rec, np.uint8)
    rows = rec.shape[:-1]
    norm, c1, cu = _unpack_polar(rec)
    bits = np.unpackbits(rec[..., 64:80][..., None], axis=-1, bitorder="little").reshape(rows + (128,))
    enorm = rec[..., 80:84].copy().view(F32).reshape(rows)
    return norm, c1, cu, bits, enorm


def decode_value64(rec):
    """Rotated-space value rows (fp64) from value records."""
    return polar_decode64(*unpack_value(rec))


def decode_key64(rec):
    """Rotated-space key rows (fp64, the PolarQuant part) and their QJL sketch."""
    norm, c1, cu, bits, enorm = unpack_key(rec)
    return polar_decode64(norm, c1, cu), bits, enorm


def compression_ratio(elt_bytes: int = 2) -> float:
    """Bytes of one token's K and V rows of one head at head_dim 128 in the
    uncompressed dtype over their records."""
    return 2 * D * elt_bytes / (KEY_BYTES + VALUE_BYTES)


# ------------------------------------------------------------------ attention
def compressed_scores(q: np.ndarray, key_recs: np.ndarray, signs, S) -> np.ndarray:
    """Estimated <q, k> / sqrt(d) for one query row q [128] against key records
    [n][96]: in the rotated space, <R q, k_hat> + the QJL estimate of <R q, e>."""
    qr = rotate64(q, signs)
    khat, bits, enorm = decode_key64(key_recs)
    return (khat @ qr + qjl_estimate(qr, bits, enorm, S)) / math.sqrt(D)


def attention_compressed(Q: np.ndarray, key_recs: np.ndarray, val_recs: np.ndarray, signs, S,
                         n_kv: int) -> np.ndarray:
    """Decode attention over compressed rows, fp64.  Q [q_len][n_q][128] are the
    last q_len positions of a sequence whose records are key_recs / val_recs
    [L][n_kv][bytes]; query j sees positions 0..L-q_len+j; query head h reads
    KV head h / (n_q / n_kv).  Softmax over the estimated scores, values
    reconstructed in the rotated space, the result rotated back."""
    Q = np.asarray(Q, np.float64)
    q_len, n_q, _ = Q.shape
    L = key_recs.shape[0]
    G = n_q // n_kv
    out = np.empty((q_len, n_q, D))
    for j in range(q_len):
        vis = L - q_len + j + 1
        for h in range(n_q):
            kv = h // G
            s = compressed_scores(Q[j, h], key_recs[:vis, kv], signs, S)
            p = np.exp(s - s.max())
            vhat = decode_value64(val_recs[:vis, kv])
            out[j, h] = unrotate64((p @ vhat) / p.sum(), signs)
    return out
