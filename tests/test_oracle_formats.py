"""Pins for the oracle's number formats (CPU only).

The e4m3 and bfloat16 codecs are checked exhaustively against PyTorch's own casts (library routines)
and against the format facts in tests/golden/e4m3_facts.txt.
"""
import os

import numpy as np
import pytest
import torch

from oracle import bf16_round, e4m3_decode, e4m3_encode_rne_satfinite
from oracle.attention import bf16_round_f64

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _facts():
    out = []
    for line in open(os.path.join(GOLDEN, "e4m3_facts.txt")):
        line = line.split("#")[0].strip()
        if line:
            c, v = line.split()
            out.append((int(c, 16), float(v)))
    return out


@pytest.mark.parametrize("code,value", _facts())
def test_e4m3_golden_facts(code, value):
    got = float(e4m3_decode(np.array([code], dtype=np.uint8))[0])
    if np.isnan(value):
        assert np.isnan(got)
    else:
        assert got == value and np.signbit(got) == np.signbit(value)


def test_e4m3_decode_exhaustive_vs_torch():
    codes = np.arange(256, dtype=np.uint8)
    ours = e4m3_decode(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    fin = ~np.isnan(ref)
    assert np.array_equal(ours[fin], ref[fin])
    assert np.array_equal(np.signbit(ours[fin]), np.signbit(ref[fin]))


def test_e4m3_plus_eight_per_doubling():
    # The property Lean P rests on: for positive normal codes, code + 8 is exactly twice the value.
    c = np.arange(8, 0x77, dtype=np.uint8)
    assert np.array_equal(e4m3_decode(c + 8), 2.0 * e4m3_decode(c))


def test_e4m3_encode_midpoints_and_random_vs_torch():
    pos = e4m3_decode(np.arange(0, 127, dtype=np.uint8))
    mids = (pos[:-1] + pos[1:]) / 2.0
    # midpoints are exact in fp32 for e4m3 neighbours, so torch's fp32 input is the same value
    rng = np.random.default_rng(3)
    rnd = rng.uniform(-448, 448, 200000)
    tiny = rng.uniform(-0.03, 0.03, 100000)
    x = np.concatenate([pos, -pos, mids, -mids, rnd, tiny]).astype(np.float32).astype(np.float64)
    ours = e4m3_encode_rne_satfinite(x)
    ref = torch.from_numpy(x.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    # both sides agree on zero's sign only up to +-0; compare values and codes away from zero
    nz = x != 0
    assert np.array_equal(ours[nz], ref[nz])


def test_e4m3_encode_saturates():
    got = e4m3_decode(e4m3_encode_rne_satfinite(np.array([448.0, 460.0, 1e6, -1e6])))
    assert list(got) == [448.0, 448.0, 448.0, -448.0]


def test_bf16_round_vs_torch():
    rng = np.random.default_rng(4)
    x = np.concatenate([rng.standard_normal(300000) * 10.0 ** rng.integers(-30, 30, 300000),
                        np.array([1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, -1.0 - 2.0 ** -8, 0.0])])
    x32 = x.astype(np.float32)
    ref = torch.from_numpy(x32).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(bf16_round(x32), ref)
    # the float64 path rounds once; on fp32-representable inputs it must agree with the fp32 path
    assert np.array_equal(bf16_round_f64(x32.astype(np.float64)), ref)
