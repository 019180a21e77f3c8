"""Pins for the Hadamard pre-pass oracle (CPU only)."""
import math
import os

import numpy as np
import pytest
import scipy.linalg

import oracle as O
from fp8_causal_prefill_gb300.inputs import Shape, make_problem

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
PAGE = {}
for line in open(os.path.join(GOLDEN, "page_figures.txt")):
    line = line.split("#")[0].strip()
    if line:
        PAGE[line.split()[0]] = float(line.split()[1])


@pytest.mark.parametrize("n", [2, 8, 64, 128])
def test_sylvester_matrix_is_scipys_hadamard(n):
    np.testing.assert_array_equal(O.hadamard_matrix(n), scipy.linalg.hadamard(n))


def test_block_sizes():
    assert O.hadamard_block(128) == 128 and O.hadamard_block(64) == 64 and O.hadamard_block(192) == 64
    with pytest.raises(ValueError):
        O.hadamard_block(96 + 1)


@pytest.mark.parametrize("d", [64, 128, 192])
def test_fast_transform_matches_the_matrix_product(d):
    rng = np.random.default_rng(d)
    x = rng.standard_normal((50, d)).astype(np.float32)
    y = O.fwht_f32(x, O.hadamard_block(d))
    ref = O.rotate(x.astype(np.float64))
    np.testing.assert_allclose(y, ref, rtol=2e-6, atol=2e-6 * np.abs(ref).max())


def test_rotation_is_orthogonal_and_an_involution():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((20, 128))
    y = O.rotate(x)
    np.testing.assert_allclose(np.linalg.norm(y, axis=1), np.linalg.norm(x, axis=1), rtol=1e-13)
    np.testing.assert_allclose(O.rotate(y), x, rtol=1e-12, atol=1e-12)


def test_exact_single_spike_maps_to_flat_row():
    # e_0 rotates to the first Hadamard column / sqrt(n): every entry +1/sqrt(n) exactly in float32
    x = np.zeros((1, 128), dtype=np.float32)
    x[0, 0] = 1.0
    y = O.fwht_f32(x, 128)
    assert np.all(y == np.float32(1.0 / math.sqrt(128)))


@pytest.mark.parametrize("d", [128, 192])
def test_attention_is_invariant_under_the_rotation(d):
    rng = np.random.default_rng(2)
    q = rng.standard_normal((1, 40, 2, d))
    k = rng.standard_normal((1, 40, 1, d))
    v = rng.standard_normal((1, 40, 1, 16))
    a = O.exact_causal_attention(q, k, v, 0.1)
    b = O.exact_causal_attention(O.rotate(q), O.rotate(k), v, 0.1)
    np.testing.assert_allclose(a, b, rtol=1e-11, atol=1e-12)


def test_quantiser_matches_the_plain_recipe_on_rotated_values():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((64, 128)).astype(np.float32)
    codes, ds = O.hadamard_quantize_e4m3(x)
    y = O.fwht_f32(x, 128)
    amax = np.float32(np.abs(y).max())
    assert ds == float(np.float32(amax / np.float32(448.0)))
    # the scale multiply agrees with the division recipe on all but a handful of boundary values
    div = O.e4m3_encode_rne_satfinite((y / np.float32(ds)).astype(np.float32).astype(np.float64))
    assert np.mean(div != codes) < 1e-3 and np.all(np.abs(div.astype(int) - codes.astype(int)) <= 1)
    assert (codes & 0x7F).max() == 0x7E                         # the maximum maps to 448
    deq = O.e4m3_decode(codes) * ds
    assert np.abs(deq).max() <= 448.0 * ds * (1 + 1e-7)
    np.testing.assert_allclose(deq, y, rtol=1.0 / 16 + 1e-6, atol=2.0 ** -9 * ds)
    z, dz = O.hadamard_quantize_e4m3(np.zeros((4, 128), dtype=np.float32))
    assert dz == 1.0 and np.all(z == 0)


def _qdq(x):
    """Per-tensor e4m3 quantise-dequantise in the original basis (the harness recipe)."""
    amax = np.float32(np.abs(x).max())
    ds = np.float32(amax / np.float32(448.0))
    return O.e4m3_decode(O.e4m3_encode_rne_satfinite((x / ds).astype(np.float32).astype(np.float64))) * ds


def _qdq_rot(x):
    """Rotate, quantise, dequantise: stays in the rotated basis (attention is invariant to it)."""
    codes, ds = O.hadamard_quantize_e4m3(x.astype(np.float32))
    return O.e4m3_decode(codes) * ds


def test_rotation_cuts_the_attention_error_from_input_quantisation():
    # The pages' figure: the rotation roughly halves the error that quantising Q and K adds.  Reading:
    # the error of the attention output against attention on the unquantised inputs (V kept exact).
    # Each e4m3 value has the same relative error in either basis; what the rotation changes is how
    # those errors add up in q.k when a few outlier channels carry most of the product.  On the
    # captured-activation stand-in (outlier channels x12) the error must fall to at most ~0.6x; on
    # plain Gaussian inputs (no outliers) there is nothing to spread and it stays within 1.15x.
    sc = 1.0 / math.sqrt(128)
    rows = np.arange(0, 1024, 7)
    for kind, bound in (("mistral", PAGE["hadamard_input_error_ratio"] + 0.1), ("gaussian", 1.15)):
        p = make_problem(Shape(1, 1024, 2, 1, 128, 128, kind), seed=0, bf16=False)
        q, k, v = p.q.astype(np.float64), p.k.astype(np.float64), p.v.astype(np.float64)
        ref = O.exact_causal_attention(q, k, v, sc, rows=rows)
        plain = O.rel_l2(O.exact_causal_attention(_qdq(q), _qdq(k), v, sc, rows=rows), ref)
        rot = O.rel_l2(O.exact_causal_attention(_qdq_rot(q), _qdq_rot(k), v, sc, rows=rows), ref)
        assert rot / plain <= bound, (kind, rot, plain)
