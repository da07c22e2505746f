"""Pins of the oracle's E4M3 codec (oracle.fp8) against the format's
definition and a library routine: printed code points of the format (1.0,
the largest finite 448, the smallest subnormal 2^-9, the smallest normal
2^-6, -2.0, NaN), decode/encode round trips over every finite code, torch's
own float8_e4m3fn cast (round to nearest even) on random in-range values,
ties to the even code, saturation beyond 448, monotonicity, and the rounding
bound of quantize/dequantize.  Planted mistakes must fail.  CPU only."""
import numpy as np
import pytest
import torch

import oracle
from oracle import fp8


def test_printed_code_points():
    assert fp8.decode([0x38])[0] == 1.0
    assert fp8.decode([0x7E])[0] == 448.0
    assert fp8.decode([0x01])[0] == 2.0 ** -9
    assert fp8.decode([0x08])[0] == 2.0 ** -6
    assert fp8.decode([0x07])[0] == 7 * 2.0 ** -9
    assert fp8.decode([0xC0])[0] == -2.0
    assert np.isnan(fp8.decode([0x7F])[0]) and np.isnan(fp8.decode([0xFF])[0])
    assert fp8.decode([0x80])[0] == 0.0 and np.signbit(fp8.decode([0x80])[0])


def test_round_trip_every_finite_code():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    np.testing.assert_array_equal(fp8.encode(fp8.decode(codes)), codes)


def test_matches_torch_cast_in_range():
    g = torch.Generator().manual_seed(5)
    x = torch.cat([torch.randn(20000, generator=g) * s for s in (1e-3, 0.05, 1.0, 30.0, 150.0)])
    x = x[x.abs() <= 448]
    ref = x.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(fp8.encode(x.numpy()), ref)


def test_ties_go_to_the_even_code_and_saturation():
    pos = fp8.decode(np.arange(127, dtype=np.uint8))
    mids = (pos[:-1] + pos[1:]) / 2
    codes = fp8.encode(mids)
    lo = np.arange(126)
    np.testing.assert_array_equal(codes, np.where(lo % 2 == 0, lo, lo + 1))
    assert fp8.encode([449.0, 1e9, -1e9])[0] == 0x7E
    assert fp8.encode([-1e9])[0] == 0xFE


def test_monotone_and_rounding_bound():
    x = np.linspace(-500, 500, 200001)
    v = fp8.decode(fp8.encode(x))
    assert np.all(np.diff(v) >= 0)
    rng = np.random.default_rng(3)
    y = rng.standard_normal(50000).astype(np.float32) * 3
    s = np.float32(0.0173)
    y = y[np.abs(y) / s <= 448]   # beyond 448 the code saturates
    d = fp8.dequantize(fp8.quantize(y, s), s)
    a = np.abs(y.astype(np.float64) / float(s))
    # half a unit in the last place of the code: 2^(e-3)/2 for normals, 2^-10 for subnormals
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -6)))
    bound = np.where(a < 2.0 ** -6, 2.0 ** -10, 2.0 ** (e - 4)) * float(s) * (1 + 1e-6)
    assert np.all(np.abs(d - y) <= bound)


def test_verify_fp8_is_verify_on_the_dequantized_history():
    rng = np.random.default_rng(9)
    B, Lmax, Hkv, D, Hq = 2, 40, 2, 16, 4
    kc = rng.integers(0, 256, size=(B, Lmax, Hkv, D)).astype(np.uint8)
    vc = rng.integers(0, 256, size=(B, Lmax, Hkv, D)).astype(np.uint8)
    kc[(kc & 0x7F) == 0x7F] = 0x3C
    vc[(vc & 0x7F) == 0x7F] = 0x3C
    ks, vs = np.array([0.01, 0.02], np.float32), np.array([0.03, 0.005], np.float32)
    cu = np.array([0, 3, 7], np.int32)
    L = np.array([30, 40], np.int32)
    q = rng.standard_normal((7, Hq, D)).astype(np.float32)
    sink = np.array([0.1, -0.5, 1.0, 0.0], np.float32)
    o = oracle.verify_fp8(q, cu, kc, vc, ks, vs, L, sink)
    kd = fp8.decode(kc) * ks[None, None, :, None].astype(np.float64)
    vd = fp8.decode(vc) * vs[None, None, :, None].astype(np.float64)
    ob = oracle.brute.verify(q, cu, kd, vd, L, sink, None, 1 / np.sqrt(D))
    np.testing.assert_allclose(o, ob, atol=1e-6)


@pytest.mark.parametrize("mutant", ["ties_away", "truncate", "bias_8", "no_saturation"])
def test_pins_reject_planted_codec_mistakes(mutant, monkeypatch):
    orig_encode, orig_pos = fp8.encode, fp8._POS.copy()

    def enc(x):
        x = np.asarray(x, np.float64)
        if mutant == "truncate":
            a = np.abs(x)
            lo = np.clip(np.searchsorted(orig_pos, a, side="right") - 1, 0, 126)
            return (lo | np.where(np.signbit(x), 0x80, 0)).astype(np.uint8)
        if mutant == "ties_away":
            return orig_encode(x * (1 + 1e-12))
        if mutant == "no_saturation":
            c = orig_encode(x)
            return np.where(np.abs(x) > 464, 0x7F | (c & 0x80), c).astype(np.uint8)
        return orig_encode(x)
    monkeypatch.setattr(fp8, "encode", enc)
    if mutant == "bias_8":
        monkeypatch.setattr(fp8, "_POS", orig_pos / 2)
    tests = [test_printed_code_points, test_round_trip_every_finite_code, test_matches_torch_cast_in_range,
             test_ties_go_to_the_even_code_and_saturation, test_monotone_and_rounding_bound]
    failed = 0
    for t in tests:
        try:
            t()
        except AssertionError:
            failed += 1
    assert failed > 0, mutant
