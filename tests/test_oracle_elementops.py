"""Pins of the oracle's element operation (no GPU).

The bf16 rounding is checked against the definition of round-to-nearest-even
evaluated independently in float64 (the two neighbouring bf16 values and their
distances), not against a second copy of the bit trick.
"""

import numpy as np
import pytest

from oracle.elementops import Arith, bf16_to_f32, f32_to_bf16_rne


def _rne_by_definition(x32):
    """Nearest bf16 to each fp32 value, ties to the even significand, chosen
    by comparing float64 distances to the two neighbours."""
    out = np.empty(x32.shape, dtype=np.uint16)
    for i, x in enumerate(x32.astype(np.float32)):
        if np.isnan(x):
            out[i] = 0x7FC0
            continue
        bits = int(np.array(x, np.float32).view(np.uint32))
        sign = bits & 0x80000000
        mag = bits & 0x7FFFFFFF
        lo = mag & 0xFFFF0000                    # toward zero
        E = (lo >> 23) & 0xFF
        if E == 0xFF:                            # infinity
            out[i] = (sign | lo) >> 16
            continue
        lo_val = float(np.array(lo, np.uint32).view(np.float32))
        ulp = 2.0 ** (max(E, 1) - 127 - 7)
        hi_val = lo_val + ulp                    # unbounded next value
        xv = abs(float(x))
        dlo, dhi = xv - lo_val, hi_val - xv
        if dlo < dhi:
            pick = lo
        elif dhi < dlo:
            pick = lo + 0x10000
        else:
            pick = lo if ((lo >> 16) & 1) == 0 else lo + 0x10000
        out[i] = (sign | pick) >> 16
    return out


def test_bf16_rne_matches_definition_random_and_edges():
    rng = np.random.default_rng(1)
    with np.errstate(over="ignore"):
        x = _draws(rng)
    x = np.concatenate([x, _tie_cases(rng)])
    got = f32_to_bf16_rne(x)
    want = _rne_by_definition(x)
    nan = np.isnan(x)
    assert np.all(np.isnan(bf16_to_f32(got[nan])))
    assert np.array_equal(got[~nan], want[~nan])


def _draws(rng):
    return np.concatenate([
        rng.standard_normal(4000).astype(np.float32),
        (rng.standard_normal(2000) * 1e-39).astype(np.float32),      # subnormal range
        (rng.standard_normal(2000) * 3e38).astype(np.float32),       # near overflow
        rng.integers(0, 2**32, 4000, dtype=np.uint64).astype(np.uint32).view(np.float32),
    ])


def _tie_cases(rng):
    # exact ties: kept part even and odd, plus values one ulp either side of a tie
    base = rng.integers(0, 0x7F7F, 500, dtype=np.uint32) << np.uint32(16)
    ties = np.concatenate([base | np.uint32(0x8000), base | np.uint32(0x7FFF),
                           base | np.uint32(0x8001)]).view(np.float32)
    special = np.array([0.0, -0.0, np.inf, -np.inf, np.nan, 3.4028235e38,
                        np.float32(np.array(0x7F7F8000, np.uint32).view(np.float32)),
                        np.float32(np.array(0x7F7F7FFF, np.uint32).view(np.float32)),
                        1e-45, -1e-45], dtype=np.float32)
    return np.concatenate([ties, special])


def test_bf16_widen_is_exact_and_roundtrips():
    allbits = np.arange(0, 2**16, dtype=np.uint32).astype(np.uint16)
    f = bf16_to_f32(allbits)
    back = f32_to_bf16_rne(f)
    finite = ~np.isnan(f)
    assert np.array_equal(back[finite], allbits[finite])


def test_bf16_sum_ties_to_even():
    # bf16 1.0 has ulp 2^-7: 1 + 2^-8 is a tie -> 1.0 (even); (1 + 2^-7) + 2^-8
    # is a tie between an odd and an even significand -> 1 + 2^-6.
    a = Arith("sum", "bfloat16")
    one = f32_to_bf16_rne(np.float32([1.0]))
    h = f32_to_bf16_rne(np.float32([2.0 ** -8]))
    odd = f32_to_bf16_rne(np.float32([1.0 + 2.0 ** -7]))
    assert bf16_to_f32(a.combine(one, h))[0] == 1.0
    assert bf16_to_f32(a.combine(odd, h))[0] == 1.0 + 2.0 ** -6


def test_int32_wraps_and_max_min_keep_right_on_ties():
    s = Arith("sum", "int32")
    assert s.combine(np.int32([2**31 - 1]), np.int32([1]))[0] == -(2**31)
    p = Arith("prod", "int32")
    assert p.combine(np.int32([65536]), np.int32([65536]))[0] == 0
    assert p.combine(np.int32([-3]), np.int32([7]))[0] == -21
    mx = Arith("max", "float32")
    pz, nz = np.float32([0.0]), np.float32([-0.0])
    assert np.signbit(mx.combine(pz, nz)[0])          # +0 > -0 is false -> right
    assert not np.signbit(mx.combine(nz, pz)[0])
    assert mx.combine(np.float32([np.nan]), np.float32([1.0]))[0] == 1.0
    assert np.isnan(mx.combine(np.float32([1.0]), np.float32([np.nan]))[0])
    mn = Arith("min", "float32")
    assert mn.combine(np.float32([2.0]), np.float32([-1.0]))[0] == -1.0


@pytest.mark.parametrize("op", ["sum", "prod", "max", "min"])
def test_bf16_op_is_fp32_op_then_rne(op):
    rng = np.random.default_rng(7)
    a = f32_to_bf16_rne(rng.standard_normal(3000).astype(np.float32))
    b = f32_to_bf16_rne(rng.standard_normal(3000).astype(np.float32))
    got = Arith(op, "bfloat16").combine(a, b)
    fa, fb = bf16_to_f32(a).astype(np.float64), bf16_to_f32(b).astype(np.float64)
    # an fp32 sum / product of two bf16 values is exact or correctly rounded;
    # computing it in float64 and rounding once to fp32 gives the same fp32
    ref = {"sum": fa + fb, "prod": fa * fb, "max": np.where(fa > fb, fa, fb),
           "min": np.where(fa < fb, fa, fb)}[op].astype(np.float32)
    assert np.array_equal(got, _rne_by_definition(ref))
