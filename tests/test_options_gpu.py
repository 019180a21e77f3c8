"""GPU parity of the options entry point (zyfa_attn_fwd_causal_ex): exact P against the exact-P
emulation (O2x), the log-sum-exp output against the oracle's, and per-(batch, KV head) descales."""
import numpy as np
import pytest
import torch

import oracle as O
from _gpu_util import BF16_TOL, FP8_TOL, per_row_rel, scale_of, select, to_device
from fp8_causal_prefill_gb300 import flash_attn_func, zyfa_check_errors
from fp8_causal_prefill_gb300.inputs import CONFIGS, Shape, make_problem, sample_rows

pytestmark = pytest.mark.gpu

SHAPES = [Shape(1, 1, 1, 1, 128, 128), Shape(1, 129, 2, 1, 128, 128), Shape(2, 520, 2, 2, 128, 128),
          Shape(1, 300, 3, 1, 64, 64), Shape(1, 513, 2, 2, 192, 128), Shape(1, 2048, 4, 1, 128, 128, "mistral")]


def _id(s):
    return f"B{s.B}S{s.S}H{s.H}kv{s.H_kv}D{s.D_qk}{'-m' if s.kind != 'gaussian' else ''}"


def _oracle(p, dtype, p_mode="lean", rows=None, heads=None):
    sc = scale_of(p)
    if dtype == "fp8":
        args = (p.q8.numpy(), p.k8.numpy(), p.v8.numpy(), p.dq, p.dk, p.dv, sc)
        f = {"exact": O.exactp_causal_attention, "exact-noblock": O.exactp_noblock_causal_attention}.get(
            p_mode, O.leanp_causal_attention)
        return f(*args, rows=rows, heads=heads, return_lse=True)
    g = lambda t: t.float().numpy().astype(np.float64)  # noqa: E731
    return O.bf16_causal_attention(g(p.qb), g(p.kb), g(p.vb), sc, rows=rows, heads=heads, return_lse=True)


def _lse_select(lse, rows=None, heads=None):
    x = lse.cpu().numpy().astype(np.float64).transpose(0, 2, 1)   # [B,S,H]
    if rows is not None:
        x = x[:, rows]
    if heads is not None:
        x = x[:, :, heads]
    return x


def _check_lse(got, ref):
    # rows agree to fp32 rounding except where an fp32 score sits on a rounding boundary of a code
    d = np.abs(got - ref)
    assert np.all(np.isfinite(got))
    assert np.median(d) <= 2e-5, np.median(d)
    assert np.mean(d <= 1e-4) >= 0.99
    assert d.max() <= 0.1


@pytest.mark.parametrize("p_mode", ["lean", "exact", "exact-noblock"])
@pytest.mark.parametrize("shape", SHAPES, ids=_id)
def test_fp8_output_and_lse_match_the_emulation(shape, p_mode):
    p = make_problem(shape, seed=shape.S + 5 * shape.H, bf16=False)
    q, k, v, ds = to_device(p, "fp8")
    out, lse = flash_attn_func(q, k, v, q_descale=ds[0], k_descale=ds[1], v_descale=ds[2], return_lse=True,
                               p_mode=p_mode)
    torch.cuda.synchronize()
    assert zyfa_check_errors() == 0
    ref, ref_lse = _oracle(p, "fp8", p_mode)
    got = select(out)
    assert O.rel_l2(got, ref) <= FP8_TOL
    assert per_row_rel(got, ref).max() <= 5e-2
    _check_lse(_lse_select(lse), ref_lse)


@pytest.mark.parametrize("shape", SHAPES[:5], ids=_id)
def test_bf16_lse_matches_the_emulation(shape):
    p = make_problem(shape, seed=shape.S + 7)
    q, k, v, _ = to_device(p, "bf16")
    out, lse = flash_attn_func(q, k, v, return_lse=True)
    torch.cuda.synchronize()
    ref, ref_lse = _oracle(p, "bf16")
    assert O.rel_l2(select(out), ref) <= BF16_TOL
    _check_lse(_lse_select(lse), ref_lse)


@pytest.mark.parametrize("p_mode", ["exact", "exact-noblock"])
def test_exact_p_full_size_sampled_rows(p_mode):
    p = make_problem(CONFIGS["bench32k"], seed=0, bf16=False)
    q, k, v, ds = to_device(p, "fp8")
    out, lse = flash_attn_func(q, k, v, q_descale=ds[0], k_descale=ds[1], v_descale=ds[2], return_lse=True,
                               p_mode=p_mode)
    torch.cuda.synchronize()
    rows = sample_rows(p.shape.S)
    heads = [0, p.shape.H - 1]
    ref, ref_lse = _oracle(p, "fp8", p_mode, rows=rows, heads=heads)
    assert O.rel_l2(select(out, rows=rows, heads=heads), ref) <= FP8_TOL
    _check_lse(_lse_select(lse, rows, heads), ref_lse)


def test_exact_p_differs_from_lean_p():
    p = make_problem(Shape(1, 700, 2, 1, 128, 128), seed=3, bf16=False)
    q, k, v, ds = to_device(p, "fp8")
    a = flash_attn_func(q, k, v, q_descale=ds[0], k_descale=ds[1], v_descale=ds[2])
    b = flash_attn_func(q, k, v, q_descale=ds[0], k_descale=ds[1], v_descale=ds[2], p_mode="exact")
    assert not torch.equal(a, b)


def test_exact_p_without_block_scaling_differs_where_blocks_lie_far_below():
    # the outlier stand-in puts many (row, block) pairs more than 8 binades below the row's reference:
    # rounding them against the reference changes the output, and each mode matches its own emulation
    p = make_problem(Shape(1, 1024, 2, 1, 128, 128, "mistral"), seed=4, bf16=False)
    q, k, v, ds = to_device(p, "fp8")
    a = flash_attn_func(q, k, v, q_descale=ds[0], k_descale=ds[1], v_descale=ds[2], p_mode="exact")
    b = flash_attn_func(q, k, v, q_descale=ds[0], k_descale=ds[1], v_descale=ds[2], p_mode="exact-noblock")
    torch.cuda.synchronize()
    assert not torch.equal(a, b)
    for mode, got in (("exact", a), ("exact-noblock", b)):
        ref, _ = _oracle(p, "fp8", mode)
        assert O.rel_l2(select(got), ref) <= FP8_TOL


def test_unknown_p_mode_is_rejected():
    p = make_problem(Shape(1, 64, 1, 1, 64, 64), seed=1, bf16=False)
    q, k, v, ds = to_device(p, "fp8")
    with pytest.raises(ValueError):
        flash_attn_func(q, k, v, p_mode="noblock")


def test_descales_per_batch_and_kv_head():
    # each (batch, KV head) gets its own q/k/v descale; the output of every head must equal the
    # oracle evaluated with that head's descales
    sh = Shape(2, 300, 4, 2, 128, 128)
    p = make_problem(sh, seed=11, bf16=False)
    rng = np.random.default_rng(12)
    dq, dk, dv = (rng.uniform(0.5, 2.0, (sh.B, sh.H_kv)).astype(np.float32) * d for d in (p.dq, p.dk, p.dv))
    q, k, v, _ = to_device(p, "fp8")
    tq, tk, tv = (torch.from_numpy(np.ascontiguousarray(x)).cuda() for x in (dq, dk, dv))
    out, lse = flash_attn_func(q, k, v, q_descale=tq, k_descale=tk, v_descale=tv, return_lse=True)
    torch.cuda.synchronize()
    got, got_lse = select(out), _lse_select(lse)
    sc = scale_of(p)
    group = sh.H // sh.H_kv
    for b in range(sh.B):
        for h in range(sh.H):
            hk = h // group
            sl = (slice(b, b + 1), slice(None), slice(h, h + 1))
            q8, k8, v8 = (t.numpy()[b:b + 1] for t in (p.q8, p.k8, p.v8))
            ref, ref_lse = O.leanp_causal_attention(q8, k8, v8, float(dq[b, hk]), float(dk[b, hk]), float(dv[b, hk]),
                                                    sc, heads=[h], return_lse=True)
            assert O.rel_l2(got[sl], ref) <= FP8_TOL
            _check_lse(got_lse[sl], ref_lse)
    # a per-tensor descale of the same value as every per-head entry gives the same bits
    one = torch.full((sh.B * sh.H_kv,), p.dq, dtype=torch.float32, device="cuda")
    onek = torch.full((sh.B * sh.H_kv,), p.dk, dtype=torch.float32, device="cuda")
    onev = torch.full((sh.B * sh.H_kv,), p.dv, dtype=torch.float32, device="cuda")
    _, _, _, ds = to_device(p, "fp8")
    a = flash_attn_func(q, k, v, q_descale=one, k_descale=onek, v_descale=onev)
    b2 = flash_attn_func(q, k, v, q_descale=ds[0], k_descale=ds[1], v_descale=ds[2])
    assert torch.equal(a, b2)
