"""Pins for the oracle's block quantiser and scalar conversions (CPU only).

Format: blocks of 32 values with one fp16 scale (Luce DFlash README,
"Asymmetric K/V quantization": q8_0 default; "Results" KV note: Q4_0 at 4.5
bits per value).  The worked examples in tests/golden/quant_examples.json were
computed by hand from the definitions.
"""
import json
import os

import numpy as np
import pytest

import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "quant_examples.json")


@pytest.fixture(scope="module")
def golden():
    with open(GOLDEN) as f:
        return json.load(f)


def _block(nonzero):
    x = np.zeros(32, np.float32)
    for j, val in nonzero.items():
        x[int(j)] = val
    return x


def test_dequant_worked_examples(orc, golden):
    for ex in golden["dequant"]:
        d16 = int(ex["d16"], 16)
        assert orc.half_to_float(d16) == ex["d"]
        if ex["type"] == "q8_0":
            qs = np.zeros(32, np.int8)
            qs[: len(ex["codes"])] = ex["codes"]
            x = orc.dequantize_q8_0(qs, d16)
        else:
            codes = np.full(32, 8, np.int64)
            codes[: len(ex["codes"])] = ex["codes"]
            nib = (codes[:16] | (codes[16:] << 4)).astype(np.uint8)
            x = orc.dequantize_q4_0(nib, d16)
        np.testing.assert_array_equal(x[: len(ex["x"])], ex["x"])


def test_quantize_worked_examples(orc, golden):
    for ex in golden["quantize"]:
        x = _block(ex["x_nonzero"])
        if ex["type"] == "q8_0":
            qs, d16 = orc.quantize_q8_0(x)
            want = np.zeros(32, np.int8)
            for j, c in ex["codes_nonzero"].items():
                want[int(j)] = c
            np.testing.assert_array_equal(qs, want)
        else:
            nib, d16 = orc.quantize_q4_0(x)
            np.testing.assert_array_equal(nib, [int(b, 16) for b in ex["bytes"]])
        assert d16 == int(ex["d16"], 16), ex["note"]


def test_bits_per_value_of_the_cache_planes(golden):
    # Bits per value of one cached row follow from the plane layout the
    # generators (and the library) use: codes plus one fp16 scale per 32.
    rng = np.random.default_rng(0)
    D = 256
    for name, t in (("q8_0", synth.KV_Q8_0), ("q4_0", synth.KV_Q4_0)):
        c = synth.kv_cache(rng, 1, 1, 4, D, t)
        row_bytes = c["kq"].shape[-1] * c["kq"].itemsize + c["ks"].shape[-1] * 2
        assert row_bytes * 8 / D == golden["bits_per_value"][name]


def test_fp16_conversion_matches_numpy(orc):
    # numpy's float32 -> float16 cast is IEEE round-to-nearest-even.
    rng = np.random.default_rng(1)
    vals = np.concatenate([
        rng.standard_normal(2000).astype(np.float32) * 10.0 ** rng.integers(-9, 5, 2000),
        np.float32([0.0, -0.0, 65504.0, 65519.0, 65520.0, 1e9, 6.1e-5, 5.96e-8, 2.98e-8,
                    2.99e-8, 1.0 + 2.0 ** -11, 1.0 + 3 * 2.0 ** -11, 2.0 ** -24 * 1.5]),
    ])
    for v in vals:
        with np.errstate(over="ignore"):
            want = int(np.float32(v).astype(np.float16).view(np.uint16))
        got = orc.float_to_half_rn(float(v))
        assert got == want, (v, hex(got), hex(want))
        if abs(v) < 65504:
            assert orc.half_to_float(got) == float(np.float16(v))


@pytest.mark.parametrize("kind", ["q8_0", "q4_0"])
def test_round_trip_error_bound(orc, kind):
    # Codes come from the fp32 scale d = amax/qmax, reconstruction uses the
    # stored fp16 d16: |x - d16 c| <= |x - d c| + |c| |d - d16| <= d/2 + qmax |d - d16|.
    rng = np.random.default_rng(2)
    qmax = 127.0 if kind == "q8_0" else 7.0
    for _ in range(300):
        x = (rng.standard_normal(32) * 10.0 ** rng.uniform(-3, 2)).astype(np.float32)
        if kind == "q8_0":
            qs, d16 = orc.quantize_q8_0(x)
            y = orc.dequantize_q8_0(qs, d16)
        else:
            nib, d16 = orc.quantize_q4_0(x)
            y = orc.dequantize_q4_0(nib, d16)
        d = float(np.abs(x).max()) / qmax
        dh = orc.half_to_float(d16)
        bound = d * (0.5 + qmax * 2.0 ** -22) + qmax * abs(d - dh) + 1e-12  # + rounding of x * (1/d)
        assert np.abs(x.astype(np.float64) - y).max() <= bound


def test_zero_block_gives_zero_scale_and_codes(orc):
    qs, d16 = orc.quantize_q8_0(np.zeros(32, np.float32))
    assert d16 == 0 and not qs.any()
    nib, d16 = orc.quantize_q4_0(np.zeros(32, np.float32))
    assert d16 == 0 and (nib == 0x88).all()


def test_divisor_examples_separate_the_two_readings(golden):
    # The quantiser could divide by the stored fp16 scale or multiply by the
    # fp32 reciprocal of the fp32 scale; both are plausible readings of the
    # format.  The examples marked with a "divided by d16" variant must give
    # different codes under the two, or they would not pin the choice.  The
    # variant is recomputed here in exact rationals (round half away).
    from fractions import Fraction

    def half_away(fr):
        return int(fr + Fraction(1, 2)) if fr >= 0 else -int(-fr + Fraction(1, 2))

    seen = 0
    for ex in golden["quantize"]:
        alt = ex.get("codes_if_divided_by_d16") or ex.get("bytes_if_divided_by_d16")
        if alt is None:
            continue
        seen += 1
        d16 = Fraction(float(np.uint16(int(ex["d16"], 16)).view(np.float16)))
        qmin, qmax = (-127, 127) if ex["type"] == "q8_0" else (-8, 7)
        codes = np.zeros(32, np.int64)
        for j, val in ex["x_nonzero"].items():
            codes[int(j)] = min(qmax, max(qmin, half_away(Fraction(val) / d16)))
        if ex["type"] == "q8_0":
            want_alt = np.zeros(32, np.int64)
            for j, c in ex["codes_if_divided_by_d16"].items():
                want_alt[int(j)] = c
            np.testing.assert_array_equal(codes, want_alt)
            want = np.zeros(32, np.int64)
            for j, c in ex["codes_nonzero"].items():
                want[int(j)] = c
            assert not np.array_equal(codes, want)
        else:
            c8 = codes + 8
            alt_bytes = (c8[:16] | (c8[16:] << 4)).astype(np.uint8)
            np.testing.assert_array_equal(alt_bytes, [int(b, 16) for b in ex["bytes_if_divided_by_d16"]])
            assert not np.array_equal(alt_bytes, [int(b, 16) for b in ex["bytes"]])
    assert seen == 2
