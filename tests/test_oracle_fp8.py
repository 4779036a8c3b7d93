"""Pins for the fp8 (E4M3) oracle: the format's definition worked by hand, exhaustive checks
over all 256 codes, round-to-nearest against brute force over every representable value,
ties to even, saturation, and the per-row quantisation's fixed points.  Planted mistakes
(ties away from zero, no saturation, a wrong subnormal step) are each caught."""
import numpy as np
import pytest

from oracle import fp8 as F

ALL = np.arange(256, dtype=np.uint8)
VALS = F.e4m3_decode(ALL)
FINITE = ~np.isnan(VALS)
GRID = np.unique(VALS[FINITE])                       # every representable value, sorted


def test_decode_by_hand():
    # sign | exponent (bias 7) | mantissa: 0x38 = 0 0111 000 = 1.0; 0x7e = 0 1111 110 = 1.75 * 2^8
    table = {0x00: 0.0, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6, 0x38: 1.0,
             0x39: 1.125, 0x3f: 1.875, 0x40: 2.0, 0x7e: 448.0, 0xb8: -1.0, 0xfe: -448.0}
    for c, v in table.items():
        assert F.e4m3_decode(np.uint8(c)) == v, hex(c)
    assert np.isnan(F.e4m3_decode(np.uint8(0x7f))) and np.isnan(F.e4m3_decode(np.uint8(0xff)))
    assert FINITE.sum() == 254
    assert GRID.max() == 448.0 and GRID[GRID > 0].min() == 2.0 ** -9


def test_code_round_trip_all_codes():
    got = F.e4m3_code(F.e4m3_round(VALS[FINITE]))
    np.testing.assert_array_equal(got, ALL[FINITE])


def test_ties_to_even_and_saturation():
    cases = {1.0625: 1.0, 1.1875: 1.25, 17.0: 16.0, 19.0: 20.0, 2.0 ** -10: 0.0,
             3 * 2.0 ** -10: 2.0 ** -8, 464.0: 448.0, 1e6: 448.0, -1e6: -448.0, -17.0: -16.0,
             0.3: 0.3125, 100.0: 96.0, 104.0: 104.0}
    for v, want in cases.items():
        assert F.e4m3_round(v) == want, (v, F.e4m3_round(v))


def test_round_to_nearest_brute_force():
    rng = np.random.default_rng(5)
    v = np.concatenate([rng.uniform(-460, 460, 4000), rng.uniform(-0.05, 0.05, 4000),
                        rng.normal(0, 3, 4000)])
    r = F.e4m3_round(v)
    d = np.abs(GRID[None, :] - np.clip(v, -448, 448)[:, None])
    best = d.min(axis=1)
    np.testing.assert_array_equal(np.abs(r - np.clip(v, -448, 448)), best)
    assert np.all(np.isin(r, GRID))
    s = np.sort(v)
    assert np.all(np.diff(F.e4m3_round(s)) >= 0)       # monotone


def test_quantize_rows_fixed_points():
    rng = np.random.default_rng(9)
    x = rng.normal(0, 2, (6, 40)).astype(np.float32)
    x[2] = 0.0
    codes, s = F.quantize_rows(x)
    assert s.dtype == np.float32 and s[2] == 1.0 and not codes[2].any()
    for i in (0, 1, 3, 4, 5):
        assert s[i] == np.float32(np.abs(x[i]).max() / np.float32(448.0))
        j = np.argmax(np.abs(x[i]))
        assert abs(F.e4m3_decode(codes[i, j])) == 448.0      # the row's amax maps to +-448
    deq = F.e4m3_decode(codes) * s[:, None]
    rel = np.abs(deq - x) / np.abs(x).max(axis=1, keepdims=True).clip(1e-30)
    assert rel.max() <= 2.0 ** -4                              # half a step of 3 mantissa bits


def test_linear_fp8_hand_worked():
    a = F.e4m3_code(np.array([[1.0, -2.0]]))
    b = F.e4m3_code(np.array([[0.5, 0.25], [3.0, 1.0]]))
    y = F.linear_fp8(a, [2.0], b, [1.0, 0.5], bias=[0.1, -1.0])
    np.testing.assert_allclose(y, [[2.0 * (0.5 - 0.5) + 0.1, 2.0 * 0.5 * (3.0 - 2.0) - 1.0]], rtol=0, atol=1e-15)


def _pins_pass():
    try:
        test_decode_by_hand()
        test_code_round_trip_all_codes()
        test_ties_to_even_and_saturation()
        test_round_to_nearest_brute_force()
        test_quantize_rows_fixed_points()
    except AssertionError:
        return False
    return True


def _ties_away(v):
    v = np.asarray(v, np.float64)
    a = np.abs(v)
    e = np.floor(np.log2(np.where(a >= F.E4M3_MIN_NORMAL, a, F.E4M3_MIN_NORMAL)))
    q = np.where(a >= F.E4M3_MIN_NORMAL, 2.0 ** (e - 3), F.E4M3_MIN_SUBNORMAL)
    return np.copysign(np.minimum(np.floor(a / q + 0.5) * q, F.E4M3_MAX), v)


ORIG = F.e4m3_round
MUTANTS = {
    "ties_away_from_zero": _ties_away,
    "no_saturation": lambda v: np.where(np.abs(np.asarray(v, np.float64)) > 448, np.asarray(v, np.float64), ORIG(v)),
    "subnormal_step_halved": lambda v: np.where(np.abs(np.asarray(v, np.float64)) < F.E4M3_MIN_NORMAL,
                                                np.round(np.asarray(v, np.float64) / 2.0 ** -10) * 2.0 ** -10,
                                                ORIG(v)),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_fp8_mistakes(name, monkeypatch):
    assert _pins_pass()
    monkeypatch.setattr(F, "e4m3_round", MUTANTS[name])
    assert not _pins_pass(), name


def test_bf16_round_by_hand():
    # 1 + 2^-8 lies halfway between 1 and 1 + 2^-7: ties to the even mantissa (1.0)
    x = np.array([1.0, 1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -9, 1.0 + 3 * 2.0 ** -8, -2.0 - 2.0 ** -7, 3.0e38])
    want = [1.0, 1.0, 1.0 + 2.0 ** -7, 1.0 + 2.0 ** -6, -2.0, 2.0 ** 127 * 1.765625]   # 3e38 = 1.7632 * 2^127
    np.testing.assert_array_equal(F.bf16_round(x), want)


def test_fp8_block_close_to_bf16_block():
    """The fp8 variant of the block equals the bf16 block up to E4M3 quantisation (a few % on
    the projections, diluted by the residual), is not the bf16 block itself, and loses its
    accuracy if the row scales are dropped."""
    import synth
    from oracle import model as M
    d = synth.Dims(hidden=128, heads=2, channels=16)
    w = synth.model_weights(d, 1, 3, bf16=True)
    bw = w.blocks[0]
    w8 = {s: F.quantize_weights(bw[s]) for s in M.STREAMS}
    rng = np.random.default_rng(2)
    xt, xi = rng.standard_normal((6, 128)), rng.standard_normal((20, 128))
    pos = M.image_positions(1, 4, 5)
    c = rng.standard_normal(128)
    ref = np.concatenate(M.block_forward(xt, xi, pos, c, bw, d.heads))
    got = np.concatenate(M.block_forward(xt, xi, pos, c, bw, d.heads, w8=w8))
    x0 = np.concatenate([xt, xi])
    dr, dg = ref - x0, got - x0
    cos = float((dr * dg).sum() / np.sqrt((dr * dr).sum() * (dg * dg).sum()))
    assert 0.99 < cos < 1.0 - 1e-9, cos
    bad = {s: dict(w8[s], s_qkv=np.ones_like(w8[s]["s_qkv"])) for s in M.STREAMS}
    gb = np.concatenate(M.block_forward(xt, xi, pos, c, bw, d.heads, w8=bad)) - x0
    cosb = float((dr * gb).sum() / np.sqrt((dr * dr).sum() * (gb * gb).sum()))
    assert cosb < 0.99, cosb
