"""Pins for O3, the compressed-row oracle (TurboQuant: PolarQuant + QJL;
dendrite demo.tape, section "TurboQuant"), against what the published
methods and the mathematics fix: the Walsh-Hadamard closed form and
orthogonality, the polar transform's geometry (bins against atan2, norms,
exact round trips of rows built from bin centres), the zero bias of the QJL
estimate, the record layout, and attention over rows that the codec
represents exactly."""
import math

import numpy as np
import pytest

from oracle import turbo_quant as T
from oracle.kv_tree import attention_dense

D = 128


def _signs(seed=0):
    return np.random.default_rng(seed).choice([-1.0, 1.0], size=D)


def test_rotation_is_the_sylvester_hadamard_matrix_with_signs():
    s = _signs(1)
    R = T.rotate64(np.eye(D), s).T               # column j = R e_j
    i, j = np.meshgrid(np.arange(D), np.arange(D), indexing="ij")
    pop = np.vectorize(lambda v: bin(v).count("1"))(i & j)
    expect = ((-1.0) ** pop) * s[None, :] / math.sqrt(D)
    assert np.allclose(R, expect, atol=1e-15)
    assert np.allclose(R @ R.T, np.eye(D), atol=1e-13)


def test_rotation_preserves_inner_products_and_inverts():
    rng = np.random.default_rng(2)
    s = _signs(2)
    x, y = rng.standard_normal((2, 5, D))
    assert np.allclose(np.sum(T.rotate64(x, s) * T.rotate64(y, s), -1), np.sum(x * y, -1), atol=1e-12)
    assert np.allclose(T.unrotate64(T.rotate64(x, s), s), x, atol=1e-13)


def test_fp32_rotation_within_rounding_of_fp64():
    rng = np.random.default_rng(3)
    s = _signs(3)
    x = rng.standard_normal((20, D)).astype(np.float32)
    err = np.abs(T.rotate32(x, s) - T.rotate64(x, s))
    # 7 rounded additions of partial sums bounded by sum|x| and one product
    bound = (8 * 2.0 ** -24) * np.abs(x).sum(-1, keepdims=True) / math.sqrt(D) + 1e-30
    assert (err <= bound).all()


def _away_from(values, boundaries, eps):
    return np.all(np.abs(values[..., None] - np.asarray(boundaries)) > eps, axis=-1)


def test_level1_codes_are_sixteenths_of_the_circle():
    rng = np.random.default_rng(4)
    a, b = rng.standard_normal((2, 20000)).astype(np.float32)
    theta = np.mod(np.arctan2(b.astype(np.float64), a.astype(np.float64)), 2 * math.pi)
    ok = _away_from(theta, np.arange(17) * math.pi / 8, 1e-5)
    x = np.zeros((20000, D), np.float32)
    x[:, 0], x[:, 1] = a, b
    x[:, 2:] = 1.0                                # the other pairs do not matter here
    _, c1, _ = T.polar_encode32(x)
    assert np.array_equal(c1[ok, 0], np.floor(theta[ok] / (math.pi / 8)).astype(np.int64))


@pytest.mark.parametrize("level", range(2, 8))
def test_upper_level_codes_are_equal_bins_of_the_level_range(level):
    lo, hi = T.upper_range(level)
    k = 2 ** (level - 1)
    assert math.isclose(hi - lo, 2 * min(math.pi / 4, 1.6 / math.sqrt(k - 1)))
    rng = np.random.default_rng(5 + level)
    n = 4000
    # a row whose level-(level) pair 0 has radii (ra, rb): put the two halves'
    # mass on one coordinate each
    phi = rng.uniform(0, math.pi / 2, size=n)
    ra, rb = np.cos(phi), np.sin(phi)
    x = np.zeros((n, D), np.float32)
    half = 2 ** (level - 1)
    x[:, 0] = ra
    x[:, half] = rb
    _, _, cu = T.polar_encode32(x)
    offs = np.cumsum([0] + [2 ** (7 - l) for l in range(2, 8)])
    code = cu[:, offs[level - 2]]
    phi32 = np.arctan2(x[:, half].astype(np.float64), x[:, 0].astype(np.float64))
    ok = _away_from(phi32, lo + np.arange(9) * (hi - lo) / 8, 1e-5)
    expect = np.clip(np.floor((phi32 - lo) / ((hi - lo) / 8)), 0, 7).astype(np.int64)
    assert np.array_equal(code[ok], expect[ok])


def test_reconstruction_keeps_the_norm_and_level1_angles_within_half_a_bin():
    rng = np.random.default_rng(6)
    x = rng.standard_normal((300, D)).astype(np.float32)
    norm, c1, cu = T.polar_encode32(x)
    xh = T.polar_decode64(norm, c1, cu)
    assert np.allclose(np.linalg.norm(xh, axis=-1), norm.astype(np.float64), rtol=1e-13)
    t_true = np.mod(np.arctan2(x[:, 1::2].astype(np.float64), x[:, 0::2].astype(np.float64)), 2 * math.pi)
    t_hat = np.mod(np.arctan2(xh[:, 1::2], xh[:, 0::2]), 2 * math.pi)
    d = np.abs(np.angle(np.exp(1j * (t_true - t_hat))))
    assert (d <= math.pi / 16 + 1e-6).all()


def test_rows_built_from_bin_centres_round_trip_exactly():
    rng = np.random.default_rng(7)
    n = 500
    c1 = rng.integers(0, 16, size=(n, 64))
    cu = rng.integers(0, 8, size=(n, 63))
    norm = rng.uniform(0.5, 20, size=n).astype(np.float32)
    x = T.polar_decode64(norm, c1, cu).astype(np.float32)
    n2, c12, cu2 = T.polar_encode32(x)
    assert np.array_equal(c12, c1) and np.array_equal(cu2, cu)
    assert np.allclose(n2, norm, rtol=1e-6)


def test_polar_error_against_fp16_rounding():
    """The reconstruction error of the 3.2x codec, next to fp16 rounding of the
    same rows (the pages' polar_vs_fp16_mae compares the two; their threshold
    is not given): on N(0, 1) rows the relative error stays below 20 %, and
    every reconstructed row is closer to its row than to any other row."""
    rng = np.random.default_rng(8)
    s = _signs(8)
    x = rng.standard_normal((400, D)).astype(np.float32)
    xr = T.rotate64(x, s)
    xh = T.polar_decode64(*T.encode_value(x, s))
    rel = np.linalg.norm(xh - xr, axis=-1) / np.linalg.norm(xr, axis=-1)
    assert rel.max() < 0.20
    mae_polar = np.abs(T.unrotate64(xh, s) - x).mean()
    mae_fp16 = np.abs(x.astype(np.float16).astype(np.float64) - x).mean()
    assert mae_fp16 < mae_polar < 0.15
    dist = np.linalg.norm(xh[:, None, :] - xr[None, :, :], axis=-1)
    assert np.array_equal(dist.argmin(axis=1), np.arange(len(x)))


def test_qjl_estimate_has_zero_bias():
    """Over random Gaussian S the estimate sqrt(pi/2)/m |e| <S q, sign(S e)>
    averages to <q, e> (the pages' qjl_zero_bias); a variant with the
    reciprocal constant does not."""
    rng = np.random.default_rng(9)
    q = rng.standard_normal(D)
    e = rng.standard_normal(D)
    ests, wrong = [], []
    for _ in range(3000):
        S = rng.standard_normal((T.M_QJL, D))
        bits = (S @ e >= 0).astype(np.uint8)
        est = T.qjl_estimate(q, bits, np.linalg.norm(e), S)
        ests.append(est)
        wrong.append(est * (2 / math.pi))
    ests = np.array(ests)
    se = ests.std() / math.sqrt(len(ests))
    assert abs(ests.mean() - q @ e) < 4 * se
    assert abs(np.mean(wrong) - q @ e) > 4 * se


def test_qjl_fp32_sketch_is_the_sign_of_the_projection():
    rng = np.random.default_rng(10)
    S = rng.standard_normal((T.M_QJL, D)).astype(np.float32)
    e = rng.standard_normal((30, D)).astype(np.float32)
    bits, enorm = T.qjl_encode32(e, S)
    z = e.astype(np.float64) @ S.T.astype(np.float64)
    clear = np.abs(z) > 1e-3
    assert np.array_equal(bits[clear], (z[clear] >= 0).astype(np.uint8))
    assert np.allclose(enorm, np.linalg.norm(e.astype(np.float64), axis=-1), rtol=1e-6)


def test_record_layout_and_ratio():
    assert T.VALUE_BYTES == 64 and T.KEY_BYTES == 96
    assert T.compression_ratio() == pytest.approx(512 / 160)
    norm = np.array([1.5], np.float32)
    c1 = np.zeros((1, 64), np.int64)
    c1[0, 0], c1[0, 1], c1[0, 63] = 3, 15, 9
    cu = np.zeros((1, 63), np.int64)
    cu[0, 0], cu[0, 1], cu[0, 62] = 5, 7, 6
    bits = np.zeros((1, 128), np.uint8)
    bits[0, 0] = bits[0, 9] = bits[0, 127] = 1
    rec = T.pack_key(norm, c1, cu, bits, np.array([2.0], np.float32))[0]
    assert rec[0:4].tobytes() == np.float32(1.5).tobytes()
    assert rec[4] == 3 | (15 << 4) and rec[35] == 9 << 4 and not rec[5:35].any()
    # 3-bit codes: 5 at bits 0..2, 7 at bits 3..5, 6 at bits 186..188
    assert rec[36] == (5 | (7 << 3)) & 0xFF and rec[37] == 7 >> 5
    assert rec[36 + 186 // 8] == (6 << (186 % 8)) & 0xFF
    assert rec[64] == 1 and rec[65] == 2 and rec[79] == 0x80
    assert rec[80:84].tobytes() == np.float32(2.0).tobytes()
    assert not rec[84:].any() and not rec[60:64].any()
    got = T.unpack_key(rec[None])
    for a, b in zip(got, (norm, c1, cu, bits, np.array([2.0], np.float32))):
        assert np.array_equal(a, b)


def test_attention_over_exactly_represented_rows_equals_dense_attention():
    """Rows built from bin centres have no residual: the codec's scores are
    the exact q.k / sqrt(d), and compressed attention equals dense softmax
    attention over the decoded rows (GQA, causal queries)."""
    rng = np.random.default_rng(11)
    s = _signs(11)
    S = rng.standard_normal((T.M_QJL, D)).astype(np.float32)
    L, n_kv, n_q, q_len = 23, 2, 4, 3

    def exact_rows():
        c1 = rng.integers(0, 16, size=(L, n_kv, 64))
        cu = rng.integers(0, 8, size=(L, n_kv, 63))
        norm = rng.uniform(5, 15, size=(L, n_kv)).astype(np.float32)
        xr = T.polar_decode64(norm, c1, cu).astype(np.float32)
        return T.unrotate64(xr, s)                  # original-space rows

    K, V = exact_rows(), exact_rows()
    keys = T.pack_key(*T.encode_key(K.astype(np.float32), s, S))
    vals = T.pack_value(*T.encode_value(V.astype(np.float32), s))
    assert np.all(T.unpack_key(keys)[4] < 1e-3)      # residual norms (fp32 rounding only)
    Q = rng.standard_normal((q_len, n_q, D))
    got = T.attention_compressed(Q, keys, vals, s, S, n_kv)
    kd = T.unrotate64(T.decode_key64(keys)[0], s)
    vd = T.unrotate64(T.decode_value64(vals), s)
    ref = attention_dense(Q, kd, vd)
    assert np.abs(got - ref).max() < 1e-3


def test_planted_quadrant_mistake_is_caught(monkeypatch):
    orig = T._bin1

    def swapped(a, b):
        return orig(b, a)
    monkeypatch.setattr(T, "_bin1", swapped)
    with pytest.raises(AssertionError):
        test_level1_codes_are_sixteenths_of_the_circle()
