"""Pins for the oracle's element formats and rounding (no GPU).

Independent references: the method statement's E2M1 value set, torch's float8_e4m3fn and bfloat16
conversions (library routines implementing IEEE round-to-nearest-even), and hand-worked ties.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle.formats import E4M3_TABLE, E2M1_TABLE

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def test_e2m1_value_set_matches_method_statement():
    assert list(oracle.E2M1_VALUES) == [0, 0.5, 1, 1.5, 2, 3, 4, 6]
    assert list(-E2M1_TABLE[8:]) == [0, 0.5, 1, 1.5, 2, 3, 4, 6]
    assert np.signbit(E2M1_TABLE[8])


def test_e4m3_decode_matches_torch_float8():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(E4M3_TABLE))
    assert np.array_equal(ref[~nan], E4M3_TABLE[~nan])
    assert oracle.E4M3_MAX == 448.0
    assert set(np.flatnonzero(nan)) == {0x7F, 0xFF}


def _torch_e4m3(v):
    return torch.from_numpy(np.asarray(v, dtype=np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_e4m3_rounding_matches_torch_on_dense_grid():
    # Every fp32 value on a dense grid of the E4M3 range, including all exact midpoints and
    # their fp32 neighbours. torch saturates nothing (it returns NaN above 464), so compare below.
    vals = np.concatenate([
        np.linspace(0, 464, 2_000_001, dtype=np.float64),
        (E4M3_TABLE[:0x7E] + E4M3_TABLE[1:0x7F]) / 2,
    ]).astype(np.float32)
    mids = vals[-0x7E:]
    vals = np.concatenate([vals, np.nextafter(mids, np.float32(0)), np.nextafter(mids, np.float32(1e9))])
    vals = vals[vals < 464]
    vals = np.concatenate([vals, -vals])
    ours = oracle.round_to_e4m3(vals.astype(np.float64))
    assert np.array_equal(ours, _torch_e4m3(vals))


def test_e4m3_rounding_subnormal_and_signed_zero():
    assert oracle.round_to_e4m3(np.array([-0.0]))[0] == 0x80
    assert oracle.round_to_e4m3(np.array([-1e-30]))[0] == 0x80
    assert oracle.round_to_e4m3(np.array([1.5 * 2 ** -9]))[0] == 0x02   # tie 1|2 -> 2
    assert oracle.round_to_e4m3(np.array([2.5 * 2 ** -9]))[0] == 0x02   # tie 2|3 -> 2
    assert oracle.round_to_e4m3(np.array([0.5 * 2 ** -9]))[0] == 0x00   # tie 0|1 -> 0
    assert oracle.round_to_e4m3(np.array([1e9]))[0] == 0x7E              # satfinite
    assert oracle.round_to_e4m3(np.array([-1e9]))[0] == 0xFE


@pytest.mark.parametrize("v,code", [
    (0.25, 0), (0.75, 2), (1.25, 2), (1.75, 4), (2.5, 4), (3.5, 6), (5.0, 6),   # ties to even
    (0.2499, 0), (0.2501, 1), (5.0001, 7), (6.0, 7), (7.0, 7), (1e30, 7),       # neighbours, sat
    (-0.25, 8), (-0.0, 8), (-3.5, 14), (-100.0, 15), (0.0, 0),
])
def test_e2m1_hand_ties(v, code):
    assert oracle.round_to_e2m1(np.array([v]))[0] == code


def test_e2m1_rounding_is_nearest_value_brute_force():
    # Brute force: nearest of the 8 magnitudes by distance, ties to the even code.
    rng = np.random.default_rng(0)
    v = np.concatenate([rng.uniform(-8, 8, 200_000), np.arange(-7, 7.01, 0.125)])
    got = oracle.round_to_e2m1(v)
    vals = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6])
    for x, g in zip(v, got):
        d = np.abs(np.abs(x) - vals)
        best = np.flatnonzero(d == d.min())
        want = best[0] if len(best) == 1 else [b for b in best if b % 2 == 0][0]
        want |= 8 if np.signbit(x) else 0
        assert g == want, (x, g, want)


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(1)
    f = np.concatenate([
        rng.standard_normal(100_000) * np.exp(rng.uniform(-90, 90, 100_000)),
        rng.standard_normal(10_000) * 2.0 ** -130,                       # bf16 subnormals
        np.array([3.3e38, -3.39e38, 3.3961e38, 0.0, -0.0, 2.0 ** -133, 2.0 ** -134]),
    ]).astype(np.float32)
    ref = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    ours = oracle.f64_to_bf16_bits_rne(f.astype(np.float64))
    assert np.array_equal(ours, ref)


def test_bf16_bits_round_trip_exhaustive():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    v = oracle.bf16_bits_to_f64(bits)
    fin = np.isfinite(v)
    assert np.array_equal(oracle.f64_to_bf16_bits_rne(v[fin]), bits[fin])
