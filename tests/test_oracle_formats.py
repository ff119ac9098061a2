"""Pins of the oracle's element codecs against the format definitions on the pages.

Each test checks the oracle against something other than itself: printed table
values, a brute-force nearest-code search, exhaustive enumeration, closed-form
bounds.
"""
import math
import random

import numpy as np
import pytest

import oracle as orc
from oracle import E2M1, E4M3, E5M2, E8M0

FMTS = {"e4m3": E4M3, "e5m2": E5M2, "e2m1": E2M1}
NBITS = {E4M3: 8, E5M2: 8, E2M1: 4}


def all_values(fmt):
    return [orc.decode(fmt, c) for c in range(1 << NBITS[fmt])]


def finite_positive(fmt):
    return sorted({v for v in all_values(fmt) if math.isfinite(v) and v > 0})


@pytest.mark.parametrize("name", ["e4m3", "e5m2"])
def test_fp8_table_values(golden, name):
    g = golden("format_limits.txt")
    fmt = FMTS[name]
    pos = finite_positive(fmt)
    assert max(pos) == float(g[(name, "max_finite")])
    assert min(pos) == float(g[(name, "min_subnormal")])
    # spacing of normal values inside [1, 2)
    in12 = [v for v in pos if 1.0 <= v < 2.0]
    steps = {b - a for a, b in zip(in12, in12[1:])}
    assert steps == {float(g[(name, "spacing_1_2")])}
    assert in12[0] == 1.0
    # smallest normal: first value whose code has a nonzero exponent field
    mbits = 3 if fmt == E4M3 else 2
    normals = [orc.decode(fmt, c) for c in range(1, 128) if (c >> mbits) != 0]
    assert min(v for v in normals if math.isfinite(v)) == float(g[(name, "min_normal")])
    if name == "e4m3":
        subn = [v for v in pos if v < float(g[(name, "min_normal")])]
        assert len(subn) == int(g[(name, "n_pos_subnormals")])


def test_e4m3_special_codes():
    # no infinities; exactly one NaN pattern per sign (S.1111.111)
    vals = all_values(E4M3)
    assert not any(math.isinf(v) for v in vals)
    nan_codes = [c for c, v in enumerate(vals) if math.isnan(v)]
    assert nan_codes == [0x7F, 0xFF]


def test_e5m2_special_codes():
    vals = all_values(E5M2)
    assert [c for c, v in enumerate(vals) if math.isinf(v)] == [0x7C, 0xFC]
    assert [c for c, v in enumerate(vals) if math.isnan(v)] == [0x7D, 0x7E, 0x7F, 0xFD, 0xFE, 0xFF]


def test_e2m1_sixteen_values(golden):
    g = golden("format_limits.txt")
    expected = [float(v) for v in g[("e2m1", "values")].split(",")]
    got = all_values(E2M1)
    assert len(got) == 16
    # the codes enumerate exactly the printed set, including both signed zeros
    assert sorted(got) == sorted(expected)
    assert [math.copysign(1, v) for v in got] == [1.0] * 8 + [-1.0] * 8
    assert max(got) == float(g[("e2m1", "max_finite")])


def test_e8m0_definition(golden):
    g = golden("format_limits.txt")
    vals = [orc.decode(E8M0, c) for c in range(256)]
    finite = [v for v in vals if math.isfinite(v)]
    assert len(finite) == 255 and sum(math.isnan(v) for v in vals) == int(g[("e8m0", "n_nan_codes")])
    ks = sorted(int(math.log2(v)) for v in finite)
    assert ks[0] == int(g[("e8m0", "k_min")]) and ks[-1] == int(g[("e8m0", "k_max")])
    assert all(v == 2.0 ** k for v, k in zip(sorted(finite), ks))


def test_emax():
    # exponent of the largest finite value: 448 = 1.75*2^8, 57344 = 1.75*2^15, 6 = 1.5*2^2
    assert orc.emax(E4M3) == 8 and orc.emax(E5M2) == 15 and orc.emax(E2M1) == 2


@pytest.mark.parametrize("fmt", [E4M3, E5M2, E2M1])
def test_roundtrip_every_finite_code(fmt):
    for c in range(1 << NBITS[fmt]):
        v = orc.decode(fmt, c)
        if math.isfinite(v):
            assert orc.encode(fmt, v) == c, (fmt, c, v)


@pytest.mark.parametrize("fmt", [E4M3, E5M2, E2M1])
def test_encode_matches_bruteforce_on_ties_and_neighbours(fmt):
    pos = finite_positive(fmt) + [0.0]
    pos = sorted(set(pos))
    probes = []
    for a, b in zip(pos, pos[1:]):
        mid = (a + b) / 2
        probes += [mid, np.nextafter(mid, 0), np.nextafter(mid, 1e300), a, b]
    top = max(pos)
    probes += [top * 1.01, top * 1.07, top * 2, 1e30, float("inf")]
    for v in probes:
        for s in (1.0, -1.0):
            x = s * float(v)
            assert orc.encode(fmt, x) == orc.encode_bruteforce(fmt, x), (fmt, x)


@pytest.mark.parametrize("fmt", [E4M3, E5M2, E2M1])
def test_encode_matches_bruteforce_random(fmt):
    rng = random.Random(1234 + fmt)
    top = max(finite_positive(fmt))
    for _ in range(3000):
        x = rng.choice([-1, 1]) * top * 2.0 ** rng.uniform(-26, 1.5)
        assert orc.encode(fmt, x) == orc.encode_bruteforce(fmt, x), (fmt, x)


def test_saturation_and_nan():
    assert orc.encode(E4M3, 460.0) == 0x7E      # rounds to 448 (480 is not a finite code)
    assert orc.encode(E4M3, 1e9) == 0x7E
    assert orc.encode(E4M3, float("inf")) == 0x7E
    assert orc.encode(E4M3, float("-inf")) == 0xFE
    assert orc.encode(E4M3, float("nan")) == 0x7F
    assert orc.encode(E5M2, float("inf")) == 0x7B
    assert orc.encode(E5M2, 70000.0) == 0x7B
    assert orc.encode(E2M1, 100.0) == 0x7
    assert orc.encode(E4M3, -0.0) == 0x80 and orc.encode(E4M3, 0.0) == 0x00
    assert orc.encode(E2M1, -0.0) == 0x8


def test_e2m1_rounding_example(golden):
    g = golden("e2m1_rounding.txt")
    x = float(g["x"])
    c = orc.encode(E2M1, x)
    q = orc.decode(E2M1, c)
    assert q == float(g["q_value"])
    assert abs(abs(q - x) / x - float(g["rel_err"])) < 1e-3


@pytest.mark.parametrize("fmt,rel", [(E4M3, "rel_err_e4m3"), (E5M2, "rel_err_e5m2")])
def test_relative_error_bound_in_normal_range(golden, fmt, rel):
    g = golden("underflow_thresholds.txt")
    bound = float(g[rel])
    pos = finite_positive(fmt)
    mbits = 3 if fmt == E4M3 else 2
    min_normal = min(orc.decode(fmt, c) for c in range(1 << mbits, 127) if math.isfinite(orc.decode(fmt, c)))
    rng = random.Random(7 + fmt)
    worst = 0.0
    for _ in range(20000):
        y = min_normal * 2.0 ** rng.uniform(0, math.log2(max(pos) / min_normal))
        q = orc.decode(fmt, orc.encode(fmt, y))
        worst = max(worst, abs(q - y) / y)
    assert worst <= bound
    # the supremum is reached just above a binade bottom: 2^-p / (1 + 2^-p)
    assert worst > 0.99 * bound / (1 + bound)


def test_span_bounds(golden):
    g = golden("underflow_thresholds.txt")
    e4 = max(finite_positive(E4M3))
    e5 = max(finite_positive(E5M2))
    min4 = 2.0 ** -6
    min5 = 2.0 ** -14
    assert e4 / min4 == float(g["full_mantissa_den"])
    assert abs(math.log2(e4 / min4) - float(g["span_log2_e4m3"])) < 0.005
    assert abs(math.log2(e5 / min5) - float(g["span_log2_e5m2"])) < 0.05
    # zero threshold: half the smallest subnormal step, relative to MAX
    assert e4 / (2.0 ** -10) == float(g["zero_den"])
