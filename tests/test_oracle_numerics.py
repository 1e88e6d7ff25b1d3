"""Oracle pins: BF16 rounding and the E4M3 codec (CPU only)."""

import numpy as np
import pytest
import torch

from oracle import numerics as nx
from oracle_pins import load_golden


def test_e4m3_decode_spec_values():
    g = load_golden("e4m3_spec_values.json")
    for c in g["decode"]:
        got = nx.e4m3_decode(np.array([int(c["code"], 16)], np.uint8))[0]
        want = float(c["value"])
        if np.isnan(want):
            assert np.isnan(got), c
        else:
            assert got == want, c


def test_e4m3_encode_spec_values():
    g = load_golden("e4m3_spec_values.json")
    for c in g["encode_rne_saturating"]:
        got = int(nx.e4m3_encode(np.array([float(c["x"])]))[0])
        assert got == int(c["code"], 16), (c, hex(got))


def test_e4m3_roundtrip_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    vals = nx.e4m3_decode(codes)
    finite = ~np.isnan(vals)
    assert finite.sum() == 254
    back = nx.e4m3_encode(vals[finite])
    assert np.array_equal(back, codes[finite])


def test_e4m3_decode_matches_torch():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = nx.e4m3_decode(codes.numpy())
    assert np.array_equal(np.isnan(ref), np.isnan(got))
    m = ~np.isnan(ref)
    assert np.array_equal(ref[m], got[m])


def test_e4m3_encode_matches_torch_cast():
    rng = np.random.default_rng(0)
    # random values over the whole range, plus every exact midpoint between
    # neighbouring codes (the ties), all inside the non-saturating range
    vals = np.concatenate([
        rng.standard_normal(20000) * 40.0,
        rng.standard_normal(20000) * 0.01,
        rng.uniform(-464, 464, 20000),
    ])
    grid = nx.e4m3_decode(np.arange(0, 0x7F, dtype=np.uint8))
    mids = (grid[:-1] + grid[1:]) / 2
    vals = np.concatenate([vals, mids, -mids, [464.0, -464.0]]).astype(np.float32)
    ref = torch.from_numpy(vals).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = nx.e4m3_encode(vals.astype(np.float64))
    assert np.array_equal(got, ref), np.flatnonzero(got != ref)[:10]


def test_e4m3_saturates_and_is_monotone():
    x = np.linspace(-2000, 2000, 100001)
    v = nx.e4m3_decode(nx.e4m3_encode(x))
    assert np.all(np.diff(v) >= 0)
    assert v.max() == 448.0 and v.min() == -448.0


def test_bf16_matches_torch_cast():
    rng = np.random.default_rng(1)
    vals = np.concatenate([
        rng.standard_normal(50000),
        rng.standard_normal(10000) * 1e-39,          # binary32 subnormals
        rng.standard_normal(10000) * 1e30,
        [3.389e38, 3.3961e38, -3.4e38, 1e-45],
    ]).astype(np.float32)
    ref = torch.from_numpy(vals).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = nx.bf16_bits(nx.bf16_round(vals.astype(np.float64)))
    assert np.array_equal(got, ref), np.flatnonzero(got != ref)[:10]


@pytest.mark.parametrize("x,want", [
    (1.0 + 2.0 ** -8, 1.0),                        # tie -> even (1.0)
    (1.0 + 3 * 2.0 ** -8, 1.0 + 2.0 ** -6),        # tie -> even (...10)
    (1.0 + 2.0 ** -8 + 2.0 ** -30, 1.0 + 2.0 ** -7),  # just above the tie
    (-(2.0 ** -133) * 1.5, -(2.0 ** -132)),        # subnormal tie -> even
])
def test_bf16_hand_ties(x, want):
    assert nx.bf16_round(np.array([x]))[0] == want


def test_bf16_bits_roundtrip():
    bits = np.arange(0, 65536, dtype=np.uint32).astype(np.uint16)
    v = nx.bf16_from_bits(bits)
    ok = np.isfinite(v)
    assert np.array_equal(nx.bf16_bits(v[ok]), bits[ok])
