"""Pins for the attention oracle (CPU only).

Each test checks the oracle against something other than itself: a figure the pages print
(tests/golden/), a closed form, an invariant of the method, a special case that reduces to a library
routine (torch's scaled_dot_product_attention / softmax), or a brute-force property on tiny inputs.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle as O
from fp8_causal_prefill_gb300.inputs import CONFIGS, Shape, far_block_fraction, make_problem, sample_rows

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_table(name):
    rows = []
    for line in open(os.path.join(GOLDEN, name)):
        line = line.split("#")[0].strip()
        if line:
            rows.append(line.split())
    return rows


PAGE = {r[0]: float(r[1]) for r in _read_table("page_figures.txt")}


def _codes(values):
    """e4m3 codes of values that must be exactly representable."""
    v = np.asarray(values, dtype=np.float64)
    c = O.e4m3_encode_rne_satfinite(v)
    assert np.array_equal(O.e4m3_decode(c), v), "test input not representable in e4m3"
    return c


def _eight_over_l8():
    """A fp32 dk with fl32(dk * fl32(8 log2 e)) == 8 exactly, so that a = 8 when scale = dq = 1."""
    l8 = np.float32(O.attention.LOG2E_X8_F32)
    base = np.float32(8.0) / l8
    for k in range(-4, 5):
        cand = np.nextafter(base, np.float32(np.inf) if k > 0 else np.float32(-np.inf)) if k else base
        for _ in range(abs(k) - 1):
            cand = np.nextafter(cand, np.float32(np.inf) if k > 0 else np.float32(-np.inf))
        if O.fp8_score_scale(1.0, 1.0, float(cand)) == 8.0:
            return float(cand)
    raise AssertionError("no fp32 dk gives a == 8")


# ----------------------------------------------------------------------------------------------
# Lean P against the pages' figures


@pytest.mark.parametrize("x,code,value", [(int(a), int(b), float(c)) for a, b, c in
                                          _read_table("leanp_integer_x.txt")])
def test_leanp_integer_powers_are_exact(x, code, value):
    got = int(O.leanp_code(np.array([8.0 * x + O.LEANP_C0]))[0])
    assert got == code == 8 * x + 56
    assert O.e4m3_decode(np.array([got], dtype=np.uint8))[0] == value == 2.0 ** x
    assert O.e4m3_encode_rne_satfinite(np.array([2.0 ** x]))[0] == code


def _leanp_rel_error(c0, xs):
    code = O.leanp_code(8.0 * xs + c0)
    return np.abs(O.e4m3_decode(code.astype(np.uint8)) - 2.0 ** xs) / 2.0 ** xs


def test_leanp_error_bound_from_pages():
    xs = np.linspace(-6.0, 0.0, 600001)
    err = _leanp_rel_error(O.LEANP_C0, xs)
    assert err.max() <= PAGE["leanp_max_rel_error"]
    assert 0.07 < err.max()                       # the bound is nearly attained (7.30%)
    exact = O.e4m3_decode(O.e4m3_encode_rne_satfinite(2.0 ** xs))
    exact_err = np.abs(exact - 2.0 ** xs) / 2.0 ** xs
    assert exact_err.max() <= PAGE["exact_rounding_max_rel_error"]
    assert abs(exact_err.max() - 1.0 / 17.0) < 1e-4   # closed form: half an ulp at mantissa 1+1/16


def test_leanp_constant_is_pinned_by_the_bound():
    # A plausible slip, c0 = 56 ("8x + 56" rounded), breaks the 7.5% figure; so does truncation.
    xs = np.linspace(-6.0, 0.0, 600001)
    assert _leanp_rel_error(56.0, xs).max() > PAGE["leanp_max_rel_error"]
    assert _leanp_rel_error(55.0, xs).max() > PAGE["leanp_max_rel_error"]


def test_leanp_block_max_lands_in_half_to_one():
    # With the block exponent e = ceil(max u / 8), the block maximum's weight is in (1/2, 1].
    rng = np.random.default_rng(0)
    s = rng.standard_normal((64, 64)) * 20
    code, e, w = O.leanp_row_weights(s, 1.0)
    blockmax_code = code.reshape(64, 1, 64).max(axis=2)
    assert np.all((blockmax_code >= 48) & (blockmax_code <= 56))


def test_leanp_shift_by_whole_binades_is_exact():
    # Shifting every score of a row by 8n code steps (n binades) must leave normalised weights
    # bit-identical: the per-block power of two absorbs the shift.
    rng = np.random.default_rng(1)
    s = np.round(rng.standard_normal((8, 300)) * 30, 2)
    _, _, w0 = O.leanp_row_weights(s, 1.0)
    for n in (-7, -1, 3, 11):
        _, e, w = O.leanp_row_weights(s + 8.0 * n, 1.0)
        assert np.array_equal(w / w.sum(1, keepdims=True), w0 / w0.sum(1, keepdims=True))


def test_block_scaling_recovers_far_blocks():
    # Worked example: keys 0..63 at probability 1, keys 64..100 ten binades lower.  Per-block
    # scaling keeps the far block exact (code 56 with scale 2^-10); a single row scale would round
    # it to code 0.
    s = np.zeros((1, 101))
    s[0, 64:] = -80.0
    code, e, w = O.leanp_row_weights(s, 1.0)
    assert list(e[0]) == [0.0, -10.0]
    assert np.all(code[0] == 56)
    assert np.all(w[0, :64] == 1.0) and np.all(w[0, 64:] == 2.0 ** -10)


def test_scale_blocks_are_64_keys_aligned_at_zero():
    # One large score at key 70 raises the exponent of keys 64..127 only.
    s = np.zeros((1, 130))
    s[0, 70] = 40.0
    _, e, w = O.leanp_row_weights(s, 1.0)
    assert list(e[0]) == [0.0, 5.0, 0.0]
    assert np.all(w[0, :64] == 2.0 ** -5) and np.all(w[0, 128:] == 2.0 ** -5)
    assert w[0, 70] == 1.0 and np.all(np.delete(w[0, 64:128], 6) == 2.0 ** -5)
    assert PAGE["scale_block_keys"] == O.SCALE_BLOCK


def test_online_tiles_match_whole_row():
    # Tiling independence: accumulate over 128-key tiles with a running integer reference M and
    # exact power-of-two rescaling, as a GPU schedule would; the result equals the whole-row oracle.
    rng = np.random.default_rng(2)
    n, d = 700, 16
    s = np.round(rng.standard_normal((4, n)) * 25, 3)
    v = O.e4m3_decode(O.e4m3_encode_rne_satfinite(rng.standard_normal((n, d))))
    _, _, w = O.leanp_row_weights(s, 1.0)
    whole = (w @ v) / w.sum(1, keepdims=True)
    for r in range(4):
        m, acc, lsum = None, np.zeros(d), 0.0
        for t0 in range(0, n, 128):
            tile = s[r, t0:t0 + 128]
            for b0 in range(0, len(tile), 64):
                blk = tile[b0:b0 + 64]
                e = math.ceil(np.max(O.fl32(blk)) / 8.0)
                if m is None or e > m:
                    if m is not None:
                        acc *= 2.0 ** (m - e)
                        lsum *= 2.0 ** (m - e)
                    m = e
                c = O.leanp_code(blk + O.LEANP_C0 - 8 * e)
                wb = O.e4m3_decode(c.astype(np.uint8)) * 2.0 ** (e - m)
                acc += wb @ v[t0 + b0:t0 + b0 + len(blk)]
                lsum += wb.sum()
        np.testing.assert_allclose(acc / lsum, whole[r], rtol=1e-14, atol=1e-14)


# ----------------------------------------------------------------------------------------------
# Whole-attention pins


def _problem_from_values(qv, kv, vv):
    q8, k8, v8 = _codes(qv), _codes(kv), _codes(vv)
    return q8, k8, v8


def test_exact_attention_matches_sdpa_with_gqa_and_mla_shape():
    rng = np.random.default_rng(5)
    b, s, h, hkv, dqk, dv = 2, 37, 4, 2, 24, 16
    q = rng.standard_normal((b, s, h, dqk))
    k = rng.standard_normal((b, s, hkv, dqk))
    v = rng.standard_normal((b, s, hkv, dv))
    sc = 0.3
    ours = O.exact_causal_attention(q, k, v, sc)
    kt = torch.from_numpy(k).repeat_interleave(h // hkv, dim=2)
    vt = torch.from_numpy(v).repeat_interleave(h // hkv, dim=2)
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q).transpose(1, 2), kt.transpose(1, 2), vt.transpose(1, 2),
        is_causal=True, scale=sc).transpose(1, 2).numpy()
    np.testing.assert_allclose(ours, ref, rtol=1e-12, atol=1e-13)


def test_base2_integer_scores_reduce_to_exact_softmax():
    # With a == 8 and integer raw scores spanning at most 6 within each 64-key block, every Lean-P code
    # is the exact e4m3 code of its probability, so O2 equals softmax in base 2 exactly.  Checked
    # against torch.softmax on scores * ln 2, with GQA and D_qk != D_v.
    rng = np.random.default_rng(6)
    b, s, h, hkv, dqk, dv = 1, 200, 4, 2, 32, 8
    # Q: one-hot rows; K: small integers whose range depends on the 64-key block, so the raw scores
    # are integers in 0..3 and the block exponents differ from block to block
    qv = np.zeros((b, s, h, dqk))
    idx = rng.integers(0, dqk, (b, s, h))
    np.put_along_axis(qv, idx[..., None], 1.0, axis=3)
    top = np.repeat(rng.integers(0, 4, (b, -(-s // 64), hkv)), 64, axis=1)[:, :s]
    kv = np.floor(rng.uniform(0, 1, (b, s, hkv, dqk)) * (top[..., None] + 1))
    vv = O.e4m3_decode(O.e4m3_encode_rne_satfinite(rng.standard_normal((b, s, hkv, dv))))
    q8, k8, v8 = _problem_from_values(qv, kv, vv)
    dk = _eight_over_l8()
    o2 = O.leanp_causal_attention(q8, k8, v8, 1.0, dk, 1.0, 1.0)
    raw = torch.einsum("bshd,bthd->bhst", torch.from_numpy(qv),
                       torch.from_numpy(kv).repeat_interleave(h // hkv, dim=2))
    assert float(raw.max() - raw.min()) <= 6.0 and len(torch.unique(raw)) == 4
    assert len(np.unique(top)) > 1
    mask = torch.ones(s, s, dtype=torch.bool).tril()
    p = torch.softmax(torch.where(mask, raw * math.log(2.0), torch.tensor(-math.inf, dtype=raw.dtype)), -1)
    ref = torch.einsum("bhst,bthd->bshd", p, torch.from_numpy(vv).repeat_interleave(h // hkv, dim=2))
    np.testing.assert_allclose(o2, ref.numpy(), rtol=1e-12, atol=1e-14)


def test_zero_queries_give_prefix_mean_on_every_path():
    # Q = 0: all scores equal, every path must return the running mean of V (closed form).
    rng = np.random.default_rng(7)
    s, dv_ = 150, 8
    q8 = np.zeros((1, s, 2, 16), dtype=np.uint8)
    k8 = O.e4m3_encode_rne_satfinite(rng.standard_normal((1, s, 1, 16)))
    vvals = O.e4m3_decode(O.e4m3_encode_rne_satfinite(rng.standard_normal((1, s, 1, dv_))))
    v8 = O.e4m3_encode_rne_satfinite(vvals)
    dv = 0.25
    mean = np.cumsum(vvals[0, :, 0, :], axis=0) / np.arange(1, s + 1)[:, None] * dv
    for f in (O.leanp_causal_attention, O.plain_fp8_causal_attention, O.exactp_noblock_causal_attention):
        out = f(q8, k8, v8, 0.5, 0.5, dv, 0.125)
        for hh in range(2):
            np.testing.assert_allclose(out[0, :, hh, :], mean, rtol=1e-14, atol=1e-15)
    ob = O.bf16_causal_attention(np.zeros((1, s, 2, 16)), O.e4m3_decode(k8), vvals * dv, 0.125)
    np.testing.assert_allclose(ob[0, :, 0, :], mean, rtol=1e-14, atol=1e-15)


def test_rounded_sum_normalisation_makes_weights_sum_to_one():
    # V == 1 everywhere: the output is sum(w)/sum(w) = 1 exactly only if the numerator and the
    # denominator use the same rounded weights (dividing by the unrounded sum would not give 1).
    p = make_problem(Shape(1, 300, 2, 1, 64, 16), seed=8, bf16=False)
    ones = np.full((1, 300, 1, 16), 0x38, dtype=np.uint8)
    out = O.leanp_causal_attention(p.q8.numpy(), p.k8.numpy(), ones, p.dq, p.dk, 1.0, 0.125)
    assert np.max(np.abs(out - 1.0)) < 1e-15
    plain = O.plain_fp8_causal_attention(p.q8.numpy(), p.k8.numpy(), ones, p.dq, p.dk, 1.0, 0.125)
    assert np.max(np.abs(plain - 1.0)) > 1e-4     # the comparator divides by the unrounded sum


def test_causality_row_zero_and_future_keys():
    p = make_problem(Shape(1, 70, 2, 2, 32, 16), seed=9)
    q8, k8, v8 = p.q8.numpy(), p.k8.numpy(), p.v8.numpy()
    args = (p.dq, p.dk, p.dv, 0.2)
    base = O.leanp_causal_attention(q8, k8, v8, *args)
    v0 = O.e4m3_decode(v8[0, 0]) * p.dv
    np.testing.assert_array_equal(base[0, 0], v0)
    pl = O.plain_fp8_causal_attention(q8, k8, v8, *args)
    np.testing.assert_array_equal(pl[0, 0], v0)
    qb, kb, vb = (t.float().numpy().astype(np.float64) for t in (p.qb, p.kb, p.vb))
    ob = O.bf16_causal_attention(qb, kb, vb, 0.2)
    np.testing.assert_array_equal(ob[0, 0], vb[0, 0])
    # perturb keys/values after row i: rows <= i must not change
    i = 40
    k2, v2 = k8.copy(), v8.copy()
    rng = np.random.default_rng(10)
    k2[:, i + 1:] = rng.integers(0, 0x7E, k2[:, i + 1:].shape, dtype=np.uint8)
    v2[:, i + 1:] = rng.integers(0, 0x7E, v2[:, i + 1:].shape, dtype=np.uint8)
    pert = O.leanp_causal_attention(q8, k2, v2, *args)
    np.testing.assert_array_equal(pert[:, :i + 1], base[:, :i + 1])
    assert not np.array_equal(pert[:, i + 1:], base[:, i + 1:])


def test_row_subset_equals_full_evaluation():
    p = make_problem(Shape(1, 333, 4, 2, 64, 64), seed=11, bf16=False)
    args = (p.q8.numpy(), p.k8.numpy(), p.v8.numpy(), p.dq, p.dk, p.dv, 0.125)
    full = O.leanp_causal_attention(*args)
    rows = np.array([0, 5, 63, 64, 65, 200, 332])
    sub = O.leanp_causal_attention(*args, rows=rows, heads=[1, 3])
    np.testing.assert_array_equal(sub, full[:, rows][:, :, [1, 3]])


def test_leanp_close_to_exact_on_gaussian():
    # Sanity bound: on Gaussian inputs Lean P stays within a few percent of float64 attention.
    p = make_problem(CONFIGS["tiny"], seed=0)
    sc = O.default_softmax_scale(64)
    q, k, v = (O.dequant_e4m3(t.numpy(), d) for t, d in ((p.q8, p.dq), (p.k8, p.dk), (p.v8, p.dv)))
    exact = O.exact_causal_attention(q, k, v, sc)
    o2 = O.leanp_causal_attention(p.q8.numpy(), p.k8.numpy(), p.v8.numpy(), p.dq, p.dk, p.dv, sc)
    o3 = O.plain_fp8_causal_attention(p.q8.numpy(), p.k8.numpy(), p.v8.numpy(), p.dq, p.dk, p.dv, sc)
    assert O.rel_l2(o2, exact) < 0.05 and O.rel_l2(o3, exact) < 0.05


def test_bf16_twin_rounded_sum_and_accuracy():
    # V == 1: the BF16 twin divides by the sum of the same rounded probabilities, so the output is 1;
    # on random bf16 inputs it stays close to float64 attention.
    rng = np.random.default_rng(12)
    s, d = 90, 16
    qb = O.bf16_round(rng.standard_normal((1, s, 1, d)))
    kb = O.bf16_round(rng.standard_normal((1, s, 1, d)))
    vb = O.bf16_round(rng.standard_normal((1, s, 1, d)))
    ones = np.ones_like(vb)
    assert np.max(np.abs(O.bf16_causal_attention(qb * 4, kb, ones, 0.25) - 1.0)) < 1e-15
    base = O.bf16_causal_attention(qb, kb, vb, 0.25)
    exact = O.exact_causal_attention(qb, kb, vb, 0.25)
    assert O.rel_l2(base, exact) < 4e-3


def test_mistral_recipe_reproduces_far_block_statistic():
    # The pages' 91% (row, 64-key block) pairs > 8 binades below the row max: the synthetic
    # stand-in must show the same property (and plain Gaussian inputs must not).
    sh = Shape(1, 2048, 4, 1, 128, 128, "mistral")
    p = make_problem(sh, seed=0, bf16=False)
    rows = np.arange(1024, 2048, 16)
    frac = far_block_fraction(p, rows, head=0)
    assert frac > PAGE["far_block_fraction"] - 0.1
    g = make_problem(Shape(1, 2048, 4, 1, 128, 128), seed=0, bf16=False)
    assert far_block_fraction(g, rows, head=0) < 0.05


def test_sample_rows_cover_edges():
    r = sample_rows(32768)
    assert r[0] == 0 and r[-1] == 32767 and len(r) == 128 * 2 + 512
    assert np.all(np.diff(r) > 0)


# ----------------------------------------------------------------------------------------------
# Exact P (the comparison the pages make for Lean P) and log-sum-exp


@pytest.mark.parametrize("x,code,value", [(int(a), int(b), float(c)) for a, b, c in
                                          _read_table("leanp_integer_x.txt")])
def test_exactp_integer_powers_match_leanp(x, code, value):
    # At whole binades both forms give the exact e4m3 code of 2^x (8x + 56).
    assert int(O.exactp_code(np.array([float(x)]))[0]) == code


def test_exactp_error_is_the_pages_exact_rounding_figure():
    t = np.linspace(-6.0, 0.0, 600001)
    code = O.exactp_code(t)
    err = np.abs(O.e4m3_decode(code.astype(np.uint8)) - 2.0 ** t) / 2.0 ** t
    assert err.max() <= PAGE["exact_rounding_max_rel_error"]
    assert abs(err.max() - 1.0 / 17.0) < 1e-4
    # and it never does worse than Lean P on the same grid
    lean = _leanp_rel_error(O.LEANP_C0, t)
    assert err.max() < lean.max()


def test_exactp_reduces_to_exact_softmax_on_integer_scores():
    # Same construction as the Lean-P case: integer base-2 scores make every probability an exact
    # power of two, so exact P, Lean P and softmax in base 2 coincide.
    rng = np.random.default_rng(6)
    b, s, h, hkv, dqk, dv = 1, 200, 4, 2, 32, 8
    qv = np.zeros((b, s, h, dqk))
    idx = rng.integers(0, dqk, (b, s, h))
    np.put_along_axis(qv, idx[..., None], 1.0, axis=3)
    top = np.repeat(rng.integers(0, 4, (b, -(-s // 64), hkv)), 64, axis=1)[:, :s]
    kv = np.floor(rng.uniform(0, 1, (b, s, hkv, dqk)) * (top[..., None] + 1))
    vv = O.e4m3_decode(O.e4m3_encode_rne_satfinite(rng.standard_normal((b, s, hkv, dv))))
    q8, k8, v8 = _problem_from_values(qv, kv, vv)
    dk = _eight_over_l8()
    ox = O.exactp_causal_attention(q8, k8, v8, 1.0, dk, 1.0, 1.0)
    o2 = O.leanp_causal_attention(q8, k8, v8, 1.0, dk, 1.0, 1.0)
    np.testing.assert_array_equal(ox, o2)
    raw = torch.einsum("bshd,bthd->bhst", torch.from_numpy(qv),
                       torch.from_numpy(kv).repeat_interleave(h // hkv, dim=2))
    mask = torch.ones(s, s, dtype=torch.bool).tril()
    p = torch.softmax(torch.where(mask, raw * math.log(2.0), torch.tensor(-math.inf, dtype=raw.dtype)), -1)
    ref = torch.einsum("bhst,bthd->bshd", p, torch.from_numpy(vv).repeat_interleave(h // hkv, dim=2))
    np.testing.assert_allclose(ox, ref.numpy(), rtol=1e-12, atol=1e-14)


def test_exactp_normalises_by_its_rounded_sum_and_differs_from_leanp():
    p = make_problem(Shape(1, 300, 2, 1, 64, 16), seed=8, bf16=False)
    ones = np.full((1, 300, 1, 16), 0x38, dtype=np.uint8)
    out = O.exactp_causal_attention(p.q8.numpy(), p.k8.numpy(), ones, p.dq, p.dk, 1.0, 0.125)
    assert np.max(np.abs(out - 1.0)) < 1e-15
    args = (p.q8.numpy(), p.k8.numpy(), p.v8.numpy(), p.dq, p.dk, p.dv, 0.125)
    assert O.rel_l2(O.exactp_causal_attention(*args), O.leanp_causal_attention(*args)) > 1e-3


def test_lse_of_exact_attention_matches_torch_logsumexp():
    rng = np.random.default_rng(13)
    b, s, h, hkv, d = 2, 45, 4, 2, 16
    q = rng.standard_normal((b, s, h, d))
    k = rng.standard_normal((b, s, hkv, d))
    v = rng.standard_normal((b, s, hkv, d))
    _, lse = O.exact_causal_attention(q, k, v, 0.4, return_lse=True)
    kt = torch.from_numpy(k).repeat_interleave(h // hkv, dim=2)
    sc = 0.4 * torch.einsum("bshd,bthd->bhst", torch.from_numpy(q), kt)
    sc = torch.where(torch.ones(s, s, dtype=torch.bool).tril(), sc, torch.tensor(-math.inf, dtype=sc.dtype))
    ref = torch.logsumexp(sc, dim=-1).permute(0, 2, 1).numpy()        # [B, S, H]
    np.testing.assert_allclose(lse, ref, rtol=1e-13, atol=1e-13)


def test_lse_of_zero_queries_is_log_of_row_length_on_every_path():
    # Q = 0: every visible score is 0, so lse_i = ln(i + 1) exactly (closed form).
    rng = np.random.default_rng(14)
    s = 130
    q8 = np.zeros((1, s, 2, 16), dtype=np.uint8)
    k8 = O.e4m3_encode_rne_satfinite(rng.standard_normal((1, s, 1, 16)))
    v8 = O.e4m3_encode_rne_satfinite(rng.standard_normal((1, s, 1, 8)))
    expect = np.log(np.arange(1, s + 1))[None, :, None]
    for f in (O.leanp_causal_attention, O.exactp_causal_attention, O.exactp_noblock_causal_attention):
        _, lse = f(q8, k8, v8, 0.5, 0.5, 1.0, 0.125, return_lse=True)
        np.testing.assert_allclose(lse, np.repeat(expect, 2, axis=2), rtol=0, atol=1e-13)
    _, lse1 = O.exact_causal_attention(np.zeros((1, s, 2, 16)), O.e4m3_decode(k8), O.e4m3_decode(v8), 0.125,
                                       return_lse=True)
    np.testing.assert_allclose(lse1, np.repeat(expect, 2, axis=2), rtol=0, atol=1e-13)
    _, lse4 = O.bf16_causal_attention(np.zeros((1, s, 2, 16)), O.e4m3_decode(k8), O.e4m3_decode(v8), 0.125,
                                      return_lse=True)
    np.testing.assert_allclose(lse4, np.repeat(expect, 2, axis=2), rtol=0, atol=1e-13)


def test_lse_of_block_scaled_paths_within_rounding_bounds_of_exact():
    # Each rounded weight is within the per-probability error bound delta of the true value, so the
    # log of their sum is within -ln(1 - delta) of the exact log-sum-exp.
    p = make_problem(Shape(1, 400, 2, 1, 64, 16), seed=15, bf16=False)
    sc = 0.125
    args = (p.q8.numpy(), p.k8.numpy(), p.v8.numpy(), p.dq, p.dk, p.dv, sc)
    q, k, v = (O.dequant_e4m3(t.numpy(), d) for t, d in ((p.q8, p.dq), (p.k8, p.dk), (p.v8, p.dv)))
    _, l1 = O.exact_causal_attention(q, k, v, sc, return_lse=True)
    _, l2 = O.leanp_causal_attention(*args, return_lse=True)
    _, lx = O.exactp_causal_attention(*args, return_lse=True)
    assert np.max(np.abs(l2 - l1)) <= -math.log1p(-PAGE["leanp_max_rel_error"])
    assert np.max(np.abs(lx - l1)) <= -math.log1p(-PAGE["exact_rounding_max_rel_error"])
    assert np.max(np.abs(l2 - l1)) > 1e-4          # the rounding is visible, not skipped


# ----------------------------------------------------------------------------------------------
# O4's rounding of each probability to bfloat16 and O2's e8m0 range, against closed forms


def _unit_bf16_scale():
    """The fp32 softmax scale whose fl32(scale * fl32(log2 e)) is exactly 1, so x = raw score."""
    sc = float(np.float32(np.float32(1.0) / np.float32(O.attention.LOG2E_F32)))
    assert O.bf16_score_scale(sc) == 1.0
    return sc


def test_bf16_twin_rounds_each_probability_to_bf16_and_uses_an_integer_reference():
    # Three rows whose scores (in binades, a' = 1) are bf16 numbers chosen so that each probability
    # 2^(x - M) falls between two bf16 values:
    #   row 1: x = [0, -127/128]: M = 0; 2^(-127/128) = 0.50271... lies between 128/256 and 129/256,
    #          nearer 129/256, so p = [1, 129/256] and with v = [0, 1] the output is 129/385;
    #   row 2: x = [-1/4, -5/4, -3]: M = ceil(-1/4) = 0 (an integer, not the row maximum);
    #          2^(-1/4) = 0.84089... -> 215/256, 2^(-5/4) = 0.42044... -> 215/512, 2^-3 = 1/8, so with
    #          v = [0, 1, 2] the output is (215/512 + 2/8) / (215/256 + 215/512 + 1/8) = 343/709.
    # Rounding p to fp32 instead, or taking M = max x, moves both outputs by more than 1e-4.
    assert 128.5 / 256 < 2 ** (-127 / 128) < 129 / 256
    assert 214.5 / 256 < 2 ** -0.25 < 215.5 / 256 and 214.5 / 512 < 2 ** -1.25 < 215.5 / 512
    sc = _unit_bf16_scale()
    d = 16
    q = np.zeros((1, 3, 1, d))
    q[0, 0, 0, 0] = q[0, 1, 0, 0] = 1.0      # rows 0 and 1 read channel 0 of the keys
    q[0, 2, 0, 1] = 1.0                      # row 2 reads channel 1
    k = np.zeros((1, 3, 1, d))
    k[0, :, 0, 0] = [0.0, -127 / 128, 0.0]
    k[0, :, 0, 1] = [-0.25, -1.25, -3.0]
    v = np.zeros((1, 3, 1, 8))
    v[0, :, 0, 0] = [0.0, 1.0, 2.0]
    v[0, :, 0, 1] = 1.0
    assert np.array_equal(O.bf16_round(np.concatenate([q.ravel(), k.ravel(), v.ravel()])),
                          np.concatenate([q.ravel(), k.ravel(), v.ravel()]))
    out = O.bf16_causal_attention(q, k, v, sc)
    assert out[0, 0, 0, 0] == 0.0
    assert abs(out[0, 1, 0, 0] - 129 / 385) < 1e-15
    assert abs(out[0, 2, 0, 0] - 343 / 709) < 1e-15
    np.testing.assert_allclose(out[0, :, 0, 1], 1.0, rtol=0, atol=1e-15)


def test_leanp_weight_is_dropped_beyond_the_e8m0_range():
    # Two 64-key blocks; the second lies 126, 127 or 130 binades below the first (a = 8, so the raw
    # score is in binades and e = ceil(score)).  Its codes are all 56 (probability 1 within the
    # block), so its weight is 2^(e_2 - e_1): kept at 2^-126, the end of the e8m0 scale range, and 0
    # beyond it.
    for below, expect in ((126, 2.0 ** -126), (127, 0.0), (130, 0.0)):
        s = np.zeros((1, 128))
        s[0, 64:] = -float(below)
        code, e, w = O.leanp_row_weights(s, 8.0)
        assert list(e[0]) == [0.0, -float(below)]
        assert np.all(code == 56) and np.all(w[0, :64] == 1.0)
        assert np.all(w[0, 64:] == expect), (below, w[0, 64])


# ----------------------------------------------------------------------------------------------
# O2xn: exact P without the per-block scaling (the ablation of the per-64-key power-of-two scaling)


def test_noblock_equals_block_scaled_when_every_block_shares_the_reference():
    # With a = 8 the exponent argument is the score itself.  Scores in (2, 3] with each 64-key block
    # reaching above 2.9: every block exponent is 3, the running reference is 3 from the first tile
    # on, so rounding against the reference is rounding against the block: O2xn == O2x, code for code.
    rng = np.random.default_rng(21)
    s32 = rng.uniform(2.01, 2.99, size=(3, 320))
    s32[:, ::64] = 2.995
    valid = np.ones(s32.shape, dtype=bool)
    c_blk, _, w_blk = O.attention._leanp_weights(s32, valid, 8.0, O.LEANP_C0, 64, exact=True)
    c_nb, m_last, w_nb = O.exactp_noblock_weights(s32, valid, 8.0)
    assert np.array_equal(m_last, np.full(3, 3.0))
    assert np.array_equal(c_nb, c_blk)
    assert np.array_equal(w_nb, w_blk)


def test_noblock_rounds_far_blocks_to_zero_where_block_scaling_keeps_them():
    # One tile: block 0 scores near 0.5 (exponent 1), block 1 scores near -11.5 (exponent -11).  Against
    # the row reference 1, 2^-12.5 lies below half the smallest e4m3 subnormal (2^-10): every code of
    # block 1 is 0, while the block-scaled path rounds 2^-0.5 and keeps weight 2^-12 per key.
    s32 = np.concatenate([np.full((1, 64), 0.5), np.full((1, 64), -11.5)], axis=1)
    valid = np.ones(s32.shape, dtype=bool)
    c_nb, _, w_nb = O.exactp_noblock_weights(s32, valid, 8.0)
    assert np.all(c_nb[0, 64:] == 0) and np.all(w_nb[0, 64:] == 0.0)
    _, _, w_blk = O.attention._leanp_weights(s32, valid, 8.0, O.LEANP_C0, 64, exact=True)
    # 2^-0.5 = 0.7071 rounds to the e4m3 value 0.6875; the block scale 2^(-11 - 1) keeps it
    np.testing.assert_array_equal(w_blk[0, 64:], np.full(64, 0.6875 * 2.0 ** -12))
    # and the output with V = 0 on block 0, 1 on block 1: 0 without block scaling, > 0 with it
    v = np.concatenate([np.zeros(64), np.ones(64)])
    assert (w_nb @ v)[0] == 0.0 and (w_blk @ v)[0] > 0.0


def test_noblock_running_reference_rises_only_beyond_eight_binades():
    # Keys 0 and 128 visible with scores t0 = 0.3 and t1; every other key far below.  Tile 0's
    # reference is ceil(0.3) = 1.
    def weights(t1):
        s32 = np.full((1, 256), -1000.0)
        s32[0, 0], s32[0, 128] = 0.3, t1
        return O.exactp_noblock_weights(s32, np.ones(s32.shape, dtype=bool), 8.0)

    # t1 = 8.5: exponent 9 = 1 + 8 is not above the threshold, the reference stays 1:
    # w1 = e4m3(2^7.5 = 181.02) = 176, w0 = e4m3(2^-0.7 = 0.6156) = 0.625
    c, m_last, w = weights(8.5)
    assert m_last[0] == 1.0
    assert (w[0, 0], w[0, 128]) == (0.625, 176.0)
    # t1 = 9.5: exponent 10 > 9, the reference becomes 10 for tile 1; tile 0's code keeps its rounding
    # against 1 and its weight is rescaled exactly: w0 = 0.625 * 2^-9, w1 = e4m3(2^-0.5) = 0.6875
    c, m_last, w = weights(9.5)
    assert m_last[0] == 10.0
    assert (w[0, 0], w[0, 128]) == (0.625 * 2.0 ** -9, 0.6875)
    # rounding tile 0 against the final reference instead would give 2^-9 (the smallest subnormal)
    assert O.e4m3_decode(O.exactp_code(np.array([0.3 - 10.0])))[0] == 2.0 ** -9


def test_noblock_later_tile_far_below_the_reference_rounds_to_zero():
    # Tile 0 sets the reference 1 (key 0 at 0.3); tile 1 lies near -11.5, below the reference, which
    # therefore does not move.  Rounded against the reference, 2^-12.5 is zero; rounded against the
    # tile's own exponent (-11) it would be e4m3(2^-0.5) = 0.6875 scaled by 2^-12.
    s32 = np.full((1, 256), -11.5)
    s32[0, 0] = 0.3
    s32[0, 1:128] = -1000.0
    c, m_last, w = O.exactp_noblock_weights(s32, np.ones(s32.shape, dtype=bool), 8.0)
    assert m_last[0] == 1.0
    assert w[0, 0] == 0.625
    assert np.all(c[0, 128:] == 0) and np.all(w[0, 128:] == 0.0)


def test_noblock_attention_is_causal_and_close_to_exact_on_gaussian():
    # Gaussian scores stay within a few binades of the row maximum, where e4m3 rounding against the
    # reference loses little: O2xn stays near float64 attention, and future keys do not matter.
    p = make_problem(Shape(1, 300, 2, 1, 64, 32), seed=22, bf16=False)
    q8, k8, v8 = p.q8.numpy(), p.k8.numpy(), p.v8.numpy()
    out = O.exactp_noblock_causal_attention(q8, k8, v8, p.dq, p.dk, p.dv, 0.125)
    ref = O.exact_causal_attention(O.dequant_e4m3(q8, p.dq), O.dequant_e4m3(k8, p.dk), O.dequant_e4m3(v8, p.dv), 0.125)
    assert O.rel_l2(out, ref) < 0.05
    k2, v2 = k8.copy(), v8.copy()
    k2[:, 200:], v2[:, 200:] = 0x38, 0x38
    out2 = O.exactp_noblock_causal_attention(q8, k2, v2, p.dq, p.dk, p.dv, 0.125)
    np.testing.assert_array_equal(out2[:, :200], out[:, :200])
